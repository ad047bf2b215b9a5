// api.cu -- the C ABI of libcredit (see include/credit.h): argument checks,
// the planner (legality + candidate choice) and dispatch to the kernels.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "credit.h"
#include "common.cuh"
#include "internal.h"
#include "planner.h"

namespace credit {

__device__ unsigned g_device_error;

#ifdef CREDIT_DEBUG
// Checked build: the per-(row, rank) combined statistics record
// (debug_row_stats); read and reset by credit_debug_stats.
__device__ float g_dbg_stats[kDbgStatsRows * kMaxCluster * kDbgStatsWidth];
#endif

// Self-test of the bounded-wait path: one thread waits on an mbarrier that
// nothing ever completes, gives up after `limit_ns` and records the timeout
// in the device error word, exactly as the kernels' waits do.  No copy is in
// flight, so the CTA exits cleanly.
__global__ void selftest_wait_kernel(unsigned* err, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    mbar_wait_limited(b, 0, err, limit_ns);
}

// A failed index check of the checked build, recorded by the same helper the
// kernels use; nothing outside any buffer is touched.
__global__ void selftest_bounds_kernel(unsigned* err) {
    __shared__ float probe[4];
    const int i = 4 + (int)threadIdx.x;  // one past the end
    if (in_bounds(i < 4, err)) probe[i] = 0.f;
}

namespace {

std::mutex g_mu;
DevInfo g_dev[kMaxDevices];
std::unordered_map<uint64_t, KernelInfo> g_kinfo;  // (device, kernel) -> info

struct DeviceGuard {  // switch device for a host query, restore on exit
    int old = -1;
    bool ok = false;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&old) != cudaSuccess) { cudaGetLastError(); return; }
        ok = old == dev || cudaSetDevice(dev) == cudaSuccess;
    }
    ~DeviceGuard() {
        if (old >= 0) cudaSetDevice(old);
    }
};

}  // namespace

const DevInfo* device_info(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    DevInfo& d = g_dev[dev];
    if (!d.valid) {
        int n = 0;
        if (cudaGetDeviceCount(&n) != cudaSuccess || dev >= n) { cudaGetLastError(); return nullptr; }
        cudaDeviceProp p;
        if (cudaGetDeviceProperties(&p, dev) != cudaSuccess) { cudaGetLastError(); return nullptr; }
        d.sms = p.multiProcessorCount;
        d.smem_optin = (int)p.sharedMemPerBlockOptin;
        d.smem_per_sm = (int)p.sharedMemPerMultiprocessor;
        d.reserved_smem = (int)p.reservedSharedMemPerBlock;
        d.l2_bytes = p.l2CacheSize;
        d.major = p.major;
        d.minor = p.minor;
        d.max_threads_sm = p.maxThreadsPerMultiProcessor;
        d.regs_per_sm = p.regsPerMultiprocessor;
        d.valid = true;
    }
    return &d;
}

// Per-(device, kernel) attributes, set once: the dynamic-SMEM opt-in up to the
// device limit and (cluster kernels) non-portable cluster sizes up to 16.
const KernelInfo* kernel_info(int dev, const void* fn, bool cluster) {
    const DevInfo* d = device_info(dev);
    if (!d || !fn) return nullptr;
    const uint64_t key = ((uint64_t)dev << 56) ^ (uint64_t)(uintptr_t)fn;
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_kinfo.find(key);
    if (it != g_kinfo.end()) return &it->second;
    DeviceGuard g(dev);
    if (!g.ok) return nullptr;
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) { cudaGetLastError(); return nullptr; }
    KernelInfo ki;
    ki.static_smem = (int)fa.sharedSizeBytes;
    ki.regs = fa.numRegs;
    ki.max_dyn_smem = d->smem_optin - ki.static_smem;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, ki.max_dyn_smem) !=
        cudaSuccess) { cudaGetLastError(); return nullptr; }
    if (cluster &&
        cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return &g_kinfo.emplace(key, ki).first->second;
}

float* debug_stats_buffer() {
#ifdef CREDIT_DEBUG
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dbg_stats) != cudaSuccess) { cudaGetLastError(); return nullptr; }
    return static_cast<float*>(p);
#else
    return nullptr;
#endif
}

unsigned* device_error_word() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) { cudaGetLastError(); return nullptr; }
    return static_cast<unsigned*>(p);
}

int occupancy_clusters(int dev, const void* fn, int P, int threads, size_t smem, int64_t rows) {
    const DevInfo* d = device_info(dev);
    if (!d) return 0;
    DeviceGuard g(dev);
    if (!g.ok) return 0;
    if (P == 1) {
        int nb = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, threads, smem) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        return nb * d->sms;
    }
    cudaLaunchConfig_t cfg = {};
    const int64_t r = std::min<int64_t>(rows, 1 << 20);
    cfg.gridDim = dim3((unsigned)(r * P), 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)P;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int nc = 0;
    if (cudaOccupancyMaxActiveClusters(&nc, fn, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return nc;
}

}  // namespace credit

using namespace credit;

namespace {

bool dtype_ok(credit_dtype_t d) { return d == CREDIT_F32 || d == CREDIT_BF16; }
size_t esize(credit_dtype_t d) { return d == CREDIT_F32 ? 4 : 2; }
bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

credit_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? CREDIT_OK : CREDIT_ERR_CUDA; }

struct OpCall {
    credit_op_t op;
    const void* x;
    void* y;
    int64_t rows, cols;
    credit_dtype_t dtype;
    const void* p0;
    const void* p1;
    credit_dtype_t pdtype;
    float eps;
    const credit_plan_t* plan;
    void* ws;
    size_t ws_bytes;
    cudaStream_t stream;
    float* aux = nullptr;  // quantization: per-row scales out
};

// Complete / re-derive a plan from the fields a caller may set.
// The L2-tail length a request asks for: its staged_elems when that is
// below its own slice_elems (a tail plan as derived) or when the request
// carries no slice_elems (a fresh request); 0 (the whole slice) otherwise,
// so a whole-slice plan stays one when its cluster size is edited.
int64_t tail_request(const credit_plan_t& r) {
    if (r.staged_elems <= 0) return 0;
    return (r.slice_elems <= 0 || r.staged_elems < r.slice_elems) ? r.staged_elems : 0;
}

credit_status_t plan_from_request(int dev, credit_op_t op, int64_t rows, int64_t cols,
                                  credit_dtype_t dtype, const credit_plan_t& r,
                                  credit_plan_t* out) {
    const credit_variant_t v = (credit_variant_t)r.variant;
    if (v != CREDIT_CLUSTER && v != CREDIT_CLUSTER_PERSISTENT && v != CREDIT_CLUSTER_PIPELINED &&
        v != CREDIT_WARP_ROWS && v != CREDIT_TWO_PASS)
        return CREDIT_ERR_INVALID_ARG;
    if (r.threads < 0 || r.ctas_per_sm < 0 || r.chunk_elems < 0 || r.rows_per_cluster < 0)
        return CREDIT_ERR_INVALID_ARG;
    const bool xok = r.exchange == CREDIT_EXCHANGE_DEFAULT ||
                     ((r.exchange == CREDIT_EXCHANGE_BARRIER || r.exchange == CREDIT_EXCHANGE_ASYNC) &&
                      v != CREDIT_TWO_PASS && v != CREDIT_WARP_ROWS);
    if (!xok) return CREDIT_ERR_INVALID_ARG;
    // the warp-specialised kernel exchanges with st.async deposits only
    if (v == CREDIT_CLUSTER_PIPELINED && r.exchange == CREDIT_EXCHANGE_BARRIER)
        return CREDIT_ERR_INVALID_ARG;
    const bool pers = v == CREDIT_CLUSTER_PERSISTENT || v == CREDIT_CLUSTER_PIPELINED;
    if (r.staged_elems < 0) return CREDIT_ERR_INVALID_ARG;
    const credit_status_t st =
        make_plan(dev, op, rows, cols, dtype, v, r.cluster_size, r.threads,
                  pers ? r.ctas_per_sm : 0, out, pers ? r.chunk_elems : 0,
                  v == CREDIT_CLUSTER ? r.rows_per_cluster : 0,
                  v == CREDIT_CLUSTER ? tail_request(r) : 0);
    if (st == CREDIT_OK && r.exchange != CREDIT_EXCHANGE_DEFAULT) out->exchange = r.exchange;
    return st;
}

// Derived launch plans, keyed by the shape and the request's fields: a call
// re-derives its plan (legality, occupancy queries) only the first time it
// sees a (device, op, shape, dtype, request) combination.  The automatic plan
// of a shape is cached too, after the profiled choice (which a later
// calibration may change) has been looked up.
struct PlanKey {
    int dev, op, dtype, variant, cluster_size, threads, cps, chunk, rpc, exchange;
    int64_t rows, cols, staged;
    bool operator==(const PlanKey& o) const {
        return std::memcmp(this, &o, sizeof(PlanKey)) == 0;
    }
};
struct PlanKeyHash {
    size_t operator()(const PlanKey& k) const {
        uint64_t h = 1469598103934665603ull;
        const unsigned char* p = reinterpret_cast<const unsigned char*>(&k);
        for (size_t i = 0; i < sizeof(PlanKey); ++i) h = (h ^ p[i]) * 1099511628211ull;
        return (size_t)h;
    }
};
std::mutex g_plan_mu;
std::unordered_map<PlanKey, credit_plan_t, PlanKeyHash> g_plans;

credit_status_t cached_plan(int dev, const OpCall& c, credit_plan_t* out) {
    credit_plan_t profiled;
    const bool automatic = !(c.plan && c.plan->variant != CREDIT_AUTO);
    const char* force = std::getenv("CREDIT_FORCE");  // a forced plan outranks a profiled one
    if (automatic && !(force && *force) &&
        lookup_profiled_plan(dev, c.op, c.rows, c.cols, c.dtype, &profiled)) {
        *out = profiled;
        return CREDIT_OK;
    }
    PlanKey k;
    std::memset(&k, 0, sizeof(k));  // no padding bytes left undefined for the hash
    k.dev = dev; k.op = (int)c.op; k.dtype = (int)c.dtype; k.rows = c.rows; k.cols = c.cols;
    if (!automatic) {
        const credit_plan_t& r = *c.plan;
        k.variant = r.variant; k.cluster_size = r.cluster_size; k.threads = r.threads;
        k.cps = r.ctas_per_sm; k.chunk = r.chunk_elems; k.rpc = r.rows_per_cluster;
        k.exchange = r.exchange; k.staged = tail_request(r);
    }
    {
        std::lock_guard<std::mutex> lk(g_plan_mu);
        auto it = g_plans.find(k);
        if (it != g_plans.end()) {
            *out = it->second;
            return CREDIT_OK;
        }
    }
    const credit_status_t st =
        automatic ? auto_plan(dev, c.op, c.rows, c.cols, c.dtype, out)
                  : plan_from_request(dev, c.op, c.rows, c.cols, c.dtype, *c.plan, out);
    if (st == CREDIT_OK) {
        std::lock_guard<std::mutex> lk(g_plan_mu);
        if (g_plans.size() >= 4096) g_plans.clear();  // bounded: shapes come and go
        g_plans.emplace(k, *out);
    }
    return st;
}

credit_status_t run(const OpCall& c) {
    if (!c.x || !c.y || c.rows < 1 || c.cols < 1) return CREDIT_ERR_INVALID_ARG;
    if (!dtype_ok(c.dtype)) return CREDIT_ERR_UNSUPPORTED;
    if ((c.p0 || c.p1) && !dtype_ok(c.pdtype)) return CREDIT_ERR_UNSUPPORTED;
    const bool quant = c.op == CREDIT_QUANTIZE;
    if (!quant && c.op != CREDIT_SOFTMAX && !(c.eps >= 0.f)) return CREDIT_ERR_INVALID_ARG;
    const bool pearson = c.op == CREDIT_PEARSON;
    if ((quant || pearson) && !c.aux) return CREDIT_ERR_INVALID_ARG;
    if ((c.op == CREDIT_WEIGHTED_STD || pearson) && !c.p0) return CREDIT_ERR_INVALID_ARG;
    if (c.rows > INT64_MAX / c.cols) return CREDIT_ERR_INVALID_ARG;
    const size_t es = esize(c.dtype);
    const int64_t n = c.rows * c.cols;
    if (n > INT64_MAX / (int64_t)es) return CREDIT_ERR_INVALID_ARG;
    // in place is fine (each element is read before it is written, by the
    // same CTA); any other overlap is rejected -- and quantization, whose
    // int8 output is narrower than its input, may not overlap at all
    const uintptr_t xb = (uintptr_t)c.x, yb = (uintptr_t)c.y;
    const uintptr_t xbytes = (uintptr_t)(n * (int64_t)es);
    const uintptr_t ybytes = quant ? (uintptr_t)n : xbytes;
    if ((quant || xb != yb) && xb < yb + ybytes && yb < xb + xbytes) return CREDIT_ERR_INVALID_ARG;
    // Pearson's second operand u has the shape of x: y may equal it (in
    // place) but may not partially overlap it
    const uintptr_t ub = pearson ? (uintptr_t)c.p0 : 0;
    if (pearson && ub != yb && ub < yb + ybytes && yb < ub + xbytes) return CREDIT_ERR_INVALID_ARG;
    if (quant || pearson) {
        const uintptr_t ab = (uintptr_t)c.aux, abytes = (uintptr_t)(c.rows * 4);
        if ((ab & 3u) || (ab < xb + xbytes && xb < ab + abytes) || (ab < yb + ybytes && yb < ab + abytes))
            return CREDIT_ERR_INVALID_ARG;
        if (pearson && ab < ub + xbytes && ub < ab + abytes) return CREDIT_ERR_INVALID_ARG;
    }

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return CREDIT_ERR_CUDA; }
    credit_plan_t plan;
    credit_status_t st;
    // a requested plan's launch shape is re-derived from (variant, P,
    // threads, ...) so a stale or hand-edited plan can never launch an
    // illegal configuration; the derivation is cached per shape and request
    st = cached_plan(dev, c, &plan);
    if (st != CREDIT_OK) return st;

    // the bulk path also needs 16-byte-aligned output rows; the int8 rows of
    // quantization are cols bytes long
    const int64_t out_row_bytes = quant ? c.cols : (int64_t)(c.cols * es);
    const bool vec = aligned16(c.x) && aligned16(c.y) && ((int64_t)(c.cols * es) % 16 == 0) &&
                     out_row_bytes % 16 == 0 && (!c.p0 || aligned16(c.p0)) &&
                     (!c.p1 || aligned16(c.p1));
    KernelKey key{(int)c.op, (int)c.dtype, (c.p0 || c.p1) ? (int)c.pdtype : 0, vec};
    unsigned* err = device_error_word();
    if (!err) return CREDIT_ERR_CUDA;
    if (!vec && plan.variant != CREDIT_TWO_PASS &&
        (plan.variant == CREDIT_CLUSTER_PERSISTENT || plan.variant == CREDIT_CLUSTER_PIPELINED ||
         plan.variant == CREDIT_WARP_ROWS || plan.rows_per_cluster != 1 ||
         (plan.staged_elems > 0 && plan.staged_elems < plan.slice_elems))) {
        // bulk copies need 16-byte alignment: misaligned or ragged rows take
        // the one-row-per-cluster kernel's element path instead, which stages
        // the whole slice (no L2 tail)
        const int32_t xchg = plan.exchange;
        st = make_plan(dev, c.op, c.rows, c.cols, c.dtype, CREDIT_CLUSTER, plan.cluster_size, 0, 0,
                       &plan, 0, 1);
        if (st != CREDIT_OK) return st;
        plan.exchange = xchg;
    }
    key.rows = plan.variant == CREDIT_CLUSTER ? plan.rows_per_cluster : 1;
    if (plan.variant == CREDIT_CLUSTER && key.rows == 1 && vec) {
        // slices too large for three CTAs per SM take the instantiation that
        // spends the spare registers on deeper parameter prefetch (where one
        // exists; cluster_kernel falls back to the regular one otherwise)
        key.deep = deep_footprint(dev, key, plan.smem_bytes);
        key.quad = quad_footprint(dev, key, plan.smem_bytes,
                                  plan.staged_elems < plan.slice_elems);
    }
    if (plan.variant == CREDIT_WARP_ROWS) {
        WarpRowsArgs a{};
        a.x = c.x; a.y = c.y; a.p0 = c.p0; a.p1 = c.p1;
        a.rows = c.rows;
        a.cols = c.cols;
        a.eps = c.eps;
        const void* fn = warp_rows_kernel(key, c.cols * (int64_t)es / 16);
        if (!fn || !kernel_info(dev, fn, false)) return CREDIT_ERR_CUDA;
        return from_cuda(launch_warp_rows(key, a, plan.active_clusters, c.stream));
    }
    if (plan.variant == CREDIT_CLUSTER_PERSISTENT || plan.variant == CREDIT_CLUSTER_PIPELINED) {
        const bool piped = plan.variant == CREDIT_CLUSTER_PIPELINED;
        PersistArgs a{};
        a.x = c.x; a.y = c.y; a.p0 = c.p0; a.p1 = c.p1;
        a.rows = c.rows;
        a.cols = c.cols;
        a.slice = (int32_t)plan.slice_elems;
        a.chunk = plan.chunk_elems;
        a.nslots = plan.ring_slots;
        a.nclusters = plan.active_clusters;
        a.eps = c.eps;
        a.err = err;
        a.exchange = (piped || plan.exchange == CREDIT_EXCHANGE_ASYNC) ? 1 : 0;
        a.dbg_stats = debug_stats_buffer();
        a.reducers = piped ? pipelined_reducers(key.op, key.dtype, plan.threads / 32 - 1) : 0;
        // the parameter room follows the ring (warp-specialised plans only)
        const int64_t ring_bytes = (int64_t)plan.ring_slots * plan.chunk_elems * (int64_t)es;
        a.param_off = piped && plan.smem_bytes > ring_bytes ? (int32_t)ring_bytes : 0;
        a.param_room = a.param_off ? (int32_t)(plan.smem_bytes - ring_bytes) : 0;
        const void* fn = piped ? pipelined_kernel(key) : persistent_kernel(key);
        if (!kernel_info(dev, fn, true)) return CREDIT_ERR_CUDA;
        return from_cuda(launch_persistent(key, a, plan.cluster_size, plan.threads,
                                           (size_t)plan.smem_bytes, c.stream));
    }

    if (plan.variant == CREDIT_CLUSTER) {
        ClusterArgs a{};
        a.x = c.x; a.y = c.y; a.p0 = c.p0; a.p1 = c.p1;
        a.rows = c.rows;
        a.cols = c.cols;
        a.slice = plan.slice_elems;
        a.chunk_elems = plan.chunk_elems;
        a.pitch = (int32_t)row_pitch(plan.staged_elems > 0 ? plan.staged_elems : plan.slice_elems,
                                     (int)es);
        a.eps = c.eps;
        a.err = err;
        a.aux = c.aux;
        a.exchange = plan.exchange == CREDIT_EXCHANGE_ASYNC ? 1 : 0;
        a.dbg_stats = debug_stats_buffer();
        a.staged = plan.staged_elems > 0 ? plan.staged_elems : plan.slice_elems;
        const void* fn = cluster_kernel(key);
        if (!kernel_info(dev, fn, true)) return CREDIT_ERR_CUDA;
        return from_cuda(launch_cluster(key, a, plan.cluster_size, plan.threads,
                                        (size_t)plan.smem_bytes, c.stream));
    }
    // two-pass baseline
    if (!c.ws || c.ws_bytes < (size_t)plan.workspace_bytes || !aligned16(c.ws))
        return CREDIT_ERR_INVALID_ARG;
    TwoPassArgs a{};
    a.x = c.x; a.y = c.y; a.p0 = c.p0; a.p1 = c.p1;
    a.cols = c.cols;
    a.chunk = (int32_t)plan.slice_elems;
    a.nch = (int32_t)((c.cols + plan.slice_elems - 1) / plan.slice_elems);
    a.eps = c.eps;
    a.ws = static_cast<float*>(c.ws);
    a.aux = c.aux;
    return from_cuda(launch_two_pass(key, a, c.rows, plan.threads, c.stream));
}

}  // namespace

extern "C" {

credit_status_t credit_plan(credit_op_t op, int64_t rows, int64_t cols, credit_dtype_t dtype,
                            int device, credit_plan_t* out) {
    if (!out) return CREDIT_ERR_INVALID_ARG;
    return auto_plan(device, op, rows, cols, dtype, out);
}

credit_status_t credit_plan_for(credit_op_t op, int64_t rows, int64_t cols, credit_dtype_t dtype,
                                int device, credit_variant_t variant, int cluster_size,
                                credit_plan_t* out) {
    if (!out) return CREDIT_ERR_INVALID_ARG;
    if (variant != CREDIT_CLUSTER && variant != CREDIT_TWO_PASS &&
        variant != CREDIT_CLUSTER_PERSISTENT && variant != CREDIT_CLUSTER_PIPELINED &&
        variant != CREDIT_WARP_ROWS)
        return CREDIT_ERR_INVALID_ARG;
    return make_plan(device, op, rows, cols, dtype, variant, cluster_size, 0, 0, out);
}

credit_status_t credit_plan_tail(credit_op_t op, int64_t rows, int64_t cols, credit_dtype_t dtype,
                                 int device, int cluster_size, int ctas_per_sm,
                                 credit_plan_t* out) {
    if (!out || rows < 1 || cols < 1 || ctas_per_sm < 1 || ctas_per_sm > 32)
        return CREDIT_ERR_INVALID_ARG;
    if (cluster_size < 1 || cluster_size > kMaxCluster) return CREDIT_ERR_NO_LEGAL_PLAN;
    if (dtype != CREDIT_F32 && dtype != CREDIT_BF16) return CREDIT_ERR_UNSUPPORTED;
    const int64_t held = tail_staged_for(device, op, cols, dtype, cluster_size, ctas_per_sm);
    if (held == 0) return CREDIT_ERR_NO_LEGAL_PLAN;
    return make_plan(device, op, rows, cols, dtype, CREDIT_CLUSTER, cluster_size, 0, 0, out, 0, 1,
                     held);
}

credit_status_t credit_plan_with(credit_op_t op, int64_t rows, int64_t cols, credit_dtype_t dtype,
                                 int device, const credit_plan_t* request, credit_plan_t* out) {
    if (!out || !request) return CREDIT_ERR_INVALID_ARG;
    return plan_from_request(device, op, rows, cols, dtype, *request, out);
}

credit_status_t credit_softmax(const void* x, void* y, int64_t rows, int64_t cols,
                               credit_dtype_t dtype, const credit_plan_t* plan, void* workspace,
                               size_t workspace_bytes, void* stream) {
    OpCall c{CREDIT_SOFTMAX, x, y, rows, cols, dtype, nullptr, nullptr, CREDIT_F32, 0.f,
             plan, workspace, workspace_bytes, (cudaStream_t)stream};
    return run(c);
}

credit_status_t credit_layernorm(const void* x, void* y, int64_t rows, int64_t cols,
                                 credit_dtype_t dtype, const void* gamma, const void* beta,
                                 credit_dtype_t param_dtype, float eps, const credit_plan_t* plan,
                                 void* workspace, size_t workspace_bytes, void* stream) {
    OpCall c{CREDIT_LAYERNORM, x, y, rows, cols, dtype, gamma, beta, param_dtype, eps,
             plan, workspace, workspace_bytes, (cudaStream_t)stream};
    return run(c);
}

credit_status_t credit_rmsnorm(const void* x, void* y, int64_t rows, int64_t cols,
                               credit_dtype_t dtype, const void* weight, credit_dtype_t param_dtype,
                               float eps, const credit_plan_t* plan, void* workspace,
                               size_t workspace_bytes, void* stream) {
    OpCall c{CREDIT_RMSNORM, x, y, rows, cols, dtype, weight, nullptr, param_dtype, eps,
             plan, workspace, workspace_bytes, (cudaStream_t)stream};
    return run(c);
}

credit_status_t credit_quantize(const void* x, int8_t* q, float* scales, int64_t rows, int64_t cols,
                                credit_dtype_t dtype, const credit_plan_t* plan, void* workspace,
                                size_t workspace_bytes, void* stream) {
    OpCall c{CREDIT_QUANTIZE, x, q, rows, cols, dtype, nullptr, nullptr, CREDIT_F32, 0.f,
             plan, workspace, workspace_bytes, (cudaStream_t)stream, scales};
    return run(c);
}

credit_status_t credit_weighted_std(const void* x, void* y, int64_t rows, int64_t cols,
                                    credit_dtype_t dtype, const void* weights,
                                    credit_dtype_t weight_dtype, float eps,
                                    const credit_plan_t* plan, void* workspace,
                                    size_t workspace_bytes, void* stream) {
    OpCall c{CREDIT_WEIGHTED_STD, x, y, rows, cols, dtype, weights, nullptr, weight_dtype, eps,
             plan, workspace, workspace_bytes, (cudaStream_t)stream};
    return run(c);
}

credit_status_t credit_pearson(const void* x, const void* u, void* y, float* r, int64_t rows,
                               int64_t cols, credit_dtype_t dtype, float eps,
                               const credit_plan_t* plan, void* workspace, size_t workspace_bytes,
                               void* stream) {
    OpCall c{CREDIT_PEARSON, x, y, rows, cols, dtype, u, nullptr, dtype, eps,
             plan, workspace, workspace_bytes, (cudaStream_t)stream, r};
    return run(c);
}

const char* credit_status_string(credit_status_t s) {
    switch (s) {
        case CREDIT_OK: return "ok";
        case CREDIT_ERR_INVALID_ARG: return "invalid argument";
        case CREDIT_ERR_UNSUPPORTED: return "unsupported dtype or op";
        case CREDIT_ERR_NO_LEGAL_PLAN: return "no legal plan (shared-memory or residency limit)";
        case CREDIT_ERR_CUDA: return "CUDA runtime error";
        case CREDIT_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait timed out";
        case CREDIT_ERR_NOT_CALIBRATED: return "device not calibrated";
        case CREDIT_ERR_DEVICE_BOUNDS: return "a device index check failed (checked build)";
    }
    return "unknown status";
}

credit_status_t credit_get_device_error(int device) {
    DeviceGuard g(device);
    if (!g.ok) return CREDIT_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) { cudaGetLastError(); return CREDIT_ERR_CUDA; }
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess) {
        cudaGetLastError();
        return CREDIT_ERR_CUDA;
    }
    if (v & kErrTimeout) return CREDIT_ERR_DEVICE_TIMEOUT;
    return (v & kErrBounds) ? CREDIT_ERR_DEVICE_BOUNDS : CREDIT_OK;
}

int credit_debug_build(void) {
#ifdef CREDIT_DEBUG
    return 1;
#else
    return 0;
#endif
}

credit_status_t credit_selftest_bounds(int device) {
#ifdef CREDIT_DEBUG
    DeviceGuard g(device);
    if (!g.ok) return CREDIT_ERR_INVALID_ARG;
    unsigned* err = device_error_word();
    if (!err) return CREDIT_ERR_CUDA;
    selftest_bounds_kernel<<<1, 1>>>(err);
    if (cudaGetLastError() != cudaSuccess) return CREDIT_ERR_CUDA;
    return credit_get_device_error(device);
#else
    (void)device;
    return CREDIT_ERR_UNSUPPORTED;
#endif
}

credit_status_t credit_debug_stats(void* host, int64_t rows) {
#ifdef CREDIT_DEBUG
    if (!host || rows < 1 || rows > kDbgStatsRows) return CREDIT_ERR_INVALID_ARG;
    const size_t bytes = (size_t)rows * kMaxCluster * kDbgStatsWidth * sizeof(float);
    float* d = debug_stats_buffer();
    if (!d || cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(host, d, bytes, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(d, 0xff, sizeof(g_dbg_stats)) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return CREDIT_ERR_CUDA;
    }
    return CREDIT_OK;
#else
    (void)host;
    (void)rows;
    return CREDIT_ERR_UNSUPPORTED;
#endif
}

credit_status_t credit_selftest_wait_timeout(int device, int64_t limit_ns) {
    if (limit_ns < 1000 || limit_ns > 1000000000) return CREDIT_ERR_INVALID_ARG;
    DeviceGuard g(device);
    if (!g.ok) return CREDIT_ERR_INVALID_ARG;
    unsigned* err = device_error_word();
    if (!err) return CREDIT_ERR_CUDA;
    selftest_wait_kernel<<<1, 1>>>(err, (unsigned long long)limit_ns);
    if (cudaGetLastError() != cudaSuccess) return CREDIT_ERR_CUDA;
    return credit_get_device_error(device);
}

const char* credit_version(void) { return "0.5.0"; }

}  // extern "C"
