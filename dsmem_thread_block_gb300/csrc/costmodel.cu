// costmodel.cu -- the profiling-fed profitability model and the per-device
// DSMEM profile it reads.
//
// CREDIT summary page (arXiv 2609.01864v1), "D. Profitability and Candidate
// Selection".  The model screens a shape with a single timing of the
// non-DSMEM path (no assumed peak bandwidth).  It prices the cluster's
// launch, scheduling, occupancy and barrier cost with a control kernel that
// does no work but has the candidate's grid, cluster size, shared-memory
// footprint and two barriers per row (T_ctrl: its time beyond the same grid
// without clusters).  It charges communication as the local replay of the
// gathered partials, the issue of the remote stores and whatever part of the
// deposits no other work hides.  The page prices the re-read that clustering
// avoids at the baseline's own rate ("D. Traffic Validation", cost
// accounting); this model uses measured local-work rates instead.
// include/credit.h has the formula as implemented.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "credit.h"
#include "common.cuh"
#include "internal.h"
#include "planner.h"

namespace credit {
namespace {

static_assert(kProfileSizes == kMaxCluster + 1, "one profile entry per cluster size");

struct DsmemProfile {
    bool valid = false;
    double barrier_ns[kMaxCluster + 1] = {};
    double exchange_ns[kMaxCluster + 1] = {};
    double async_exchange_ns[kMaxCluster + 1] = {};
    double local_load_ns = 0.0;  // one shared-memory hop: the local replay's unit
};

std::mutex g_cm_mu;
DsmemProfile g_profile[kMaxDevices];
std::map<std::tuple<int, int, int, int64_t, int64_t>, credit_plan_t> g_chosen;
// local-work primitive rates per (device, op, dtype, parameter dtype)
std::map<std::tuple<int, int, int, int>, LocalRates> g_local;

int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct Scratch {
    void* p = nullptr;
    ~Scratch() { if (p) cudaFree(p); }
    bool alloc(size_t n) {
        if (n == 0) return true;
        if (cudaMalloc(&p, n) != cudaSuccess) { cudaGetLastError(); p = nullptr; return false; }
        return cudaMemset(p, 0, n) == cudaSuccess;
    }
};

// Timing inputs: values spread uniformly over [lo, hi) from an integer hash
// of the index (Wellons' "lowbias32" mixer), so the kernels are timed on
// varied data -- constant zeros would skip work (an all-zero quantization row
// divides nothing; a constant softmax row never rescales).
__device__ __forceinline__ uint32_t mix32(uint32_t x) {
    x ^= x >> 16;
    x *= 0x7feb352du;
    x ^= x >> 15;
    x *= 0x846ca68bu;
    x ^= x >> 16;
    return x;
}

__global__ void fill_kernel(void* p, int64_t n, int bf16, float lo, float hi, uint32_t seed) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const uint32_t h = mix32((uint32_t)i ^ mix32((uint32_t)(i >> 32) ^ seed));
        const float v = lo + (hi - lo) * (float)(h >> 8) * (1.0f / 16777216.0f);
        if (bf16) static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
        else static_cast<float*>(p)[i] = v;
    }
}

bool fill(void* p, int64_t n, credit_dtype_t dt, float lo, float hi, uint32_t seed) {
    if (!p || n == 0) return true;
    fill_kernel<<<1024, 256>>>(p, n, dt == CREDIT_BF16 ? 1 : 0, lo, hi, seed);
    return cudaGetLastError() == cudaSuccess;
}

double median_of(std::vector<double> v) {
    std::sort(v.begin(), v.end());
    const size_t n = v.size();
    return n % 2 ? v[n / 2] : 0.5 * (v[n / 2 - 1] + v[n / 2]);
}

}  // namespace

bool lookup_profiled_plan(int dev, credit_op_t op, int64_t rows, int64_t cols,
                          credit_dtype_t dtype, credit_plan_t* out) {
    profile_env_load(dev);  // CREDIT_PROFILE: the saved choices, once per device
    std::lock_guard<std::mutex> lk(g_cm_mu);
    auto it = g_chosen.find(std::make_tuple(dev, (int)op, (int)dtype, rows, cols));
    if (it == g_chosen.end()) return false;
    *out = it->second;
    return true;
}

bool dsmem_profile_get(int dev, DsmemData* out) {
    if (dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lk(g_cm_mu);
    const DsmemProfile& p = g_profile[dev];
    if (!p.valid) return false;
    for (int P = 0; P <= kMaxCluster; ++P) {
        out->barrier_ns[P] = p.barrier_ns[P];
        out->exchange_ns[P] = p.exchange_ns[P];
        out->async_ns[P] = p.async_exchange_ns[P];
    }
    out->local_load_ns = p.local_load_ns;
    return true;
}

void dsmem_profile_set(int dev, const DsmemData& d) {
    if (dev < 0 || dev >= kMaxDevices) return;
    DsmemProfile p;
    for (int P = 0; P <= kMaxCluster; ++P) {
        p.barrier_ns[P] = d.barrier_ns[P];
        p.exchange_ns[P] = d.exchange_ns[P];
        p.async_exchange_ns[P] = d.async_ns[P];
    }
    p.local_load_ns = d.local_load_ns;
    p.valid = true;
    std::lock_guard<std::mutex> lk(g_cm_mu);
    g_profile[dev] = p;
}

std::vector<LocalRates> local_rates(int dev) {
    std::vector<LocalRates> out;
    std::lock_guard<std::mutex> lk(g_cm_mu);
    for (const auto& kv : g_local)
        if (std::get<0>(kv.first) == dev) out.push_back(kv.second);
    return out;
}

void local_rates_put(int dev, const LocalRates& r) {
    std::lock_guard<std::mutex> lk(g_cm_mu);
    g_local[std::make_tuple(dev, r.op, r.dtype, r.pdt)] = r;
}

std::vector<ChosenPlan> chosen_plans(int dev) {
    std::vector<ChosenPlan> out;
    std::lock_guard<std::mutex> lk(g_cm_mu);
    for (const auto& kv : g_chosen) {
        if (std::get<0>(kv.first) != dev) continue;
        out.push_back(ChosenPlan{std::get<1>(kv.first), std::get<2>(kv.first),
                                 std::get<3>(kv.first), std::get<4>(kv.first), kv.second});
    }
    return out;
}

void chosen_plan_put(int dev, const ChosenPlan& c) {
    std::lock_guard<std::mutex> lk(g_cm_mu);
    g_chosen[std::make_tuple(dev, c.op, c.dtype, c.rows, c.cols)] = c.plan;
}

}  // namespace credit

using namespace credit;

extern "C" credit_status_t credit_calibrate(int device, int runs, const char* profile_path) {
    if (device < 0 || device >= kMaxDevices || runs < 1) return CREDIT_ERR_INVALID_ARG;
    // CREDIT_PROFILE: read what the file already holds first, so the write
    // below keeps it (plans and primitive rates) instead of replacing it
    profile_env_load(device);
    DsmemProfile prof;
    for (int P = 2; P <= kMaxCluster; ++P) {
        credit_bench_result_t b, e, x;
        credit_status_t st = credit_bench_dsmem(device, CREDIT_BENCH_BARRIER, P, 500, runs, &b);
        if (st != CREDIT_OK) return st;
        st = credit_bench_dsmem(device, CREDIT_BENCH_EXCHANGE, P, 500, runs, &e);
        if (st != CREDIT_OK) return st;
        st = credit_bench_dsmem(device, CREDIT_BENCH_ASYNC_EXCHANGE, P, 500, runs, &x);
        if (st != CREDIT_OK) return st;
        prof.barrier_ns[P] = b.median_ns;
        prof.exchange_ns[P] = e.median_ns;
        prof.async_exchange_ns[P] = x.median_ns;
    }
    {
        credit_bench_result_t l;
        const credit_status_t st =
            credit_bench_dsmem(device, CREDIT_BENCH_LOCAL_LOAD_LATENCY, 2, 2000, runs, &l);
        if (st != CREDIT_OK) return st;
        prof.local_load_ns = l.median_ns;
    }
    prof.valid = true;
    {
        std::lock_guard<std::mutex> lk(g_cm_mu);
        g_profile[device] = prof;
    }
    if (profile_path) {
        const credit_status_t st = credit_save_profile(device, profile_path);
        if (st != CREDIT_OK) return st;
    }
    profile_env_save(device);
    return CREDIT_OK;
}

namespace {

// One launch of the operator with an explicit plan on the default stream
// (aux: the row scales of quantization).
credit_status_t call_op(credit_op_t op, const void* x, void* y, int64_t rows, int64_t cols,
                        credit_dtype_t dtype, const void* p0, const void* p1, int pdt,
                        const credit_plan_t* plan, void* ws, size_t wsb, float* aux) {
    const credit_dtype_t pd = pdt < 0 ? CREDIT_F32 : (credit_dtype_t)pdt;
    switch (op) {
        case CREDIT_QUANTIZE:
            return credit_quantize(x, static_cast<int8_t*>(y), aux, rows, cols, dtype, plan, ws, wsb,
                                   nullptr);
        case CREDIT_WEIGHTED_STD:
            return credit_weighted_std(x, y, rows, cols, dtype, p0, pd, 1e-5f, plan, ws, wsb,
                                       nullptr);
        case CREDIT_PEARSON:
            return credit_pearson(x, p0, y, aux, rows, cols, dtype, 1e-5f, plan, ws, wsb, nullptr);
        case CREDIT_SOFTMAX: return credit_softmax(x, y, rows, cols, dtype, plan, ws, wsb, nullptr);
        case CREDIT_LAYERNORM:
            return credit_layernorm(x, y, rows, cols, dtype, p0, p1, pd, 1e-5f, plan, ws, wsb, nullptr);
        case CREDIT_RMSNORM:
            return credit_rmsnorm(x, y, rows, cols, dtype, p0, pd, 1e-6f, plan, ws, wsb, nullptr);
    }
    return CREDIT_ERR_UNSUPPORTED;
}

// Median time of `runs` launches (after one warm-up) in microseconds.
credit_status_t time_op(credit_op_t op, const void* x, void* y, int64_t rows, int64_t cols,
                        credit_dtype_t dtype, const void* p0, const void* p1, int pdt,
                        const credit_plan_t* plan, void* ws, size_t wsb, int runs, double* us,
                        float* aux) {
    cudaEvent_t e0, e1;
    if (cudaEventCreate(&e0) != cudaSuccess) return CREDIT_ERR_CUDA;
    if (cudaEventCreate(&e1) != cudaSuccess) { cudaEventDestroy(e0); return CREDIT_ERR_CUDA; }
    std::vector<double> t;
    credit_status_t st = CREDIT_OK;
    for (int r = 0; r <= runs && st == CREDIT_OK; ++r) {
        float ms = 0.f;
        if (cudaEventRecord(e0, nullptr) != cudaSuccess) { st = CREDIT_ERR_CUDA; break; }
        st = call_op(op, x, y, rows, cols, dtype, p0, p1, pdt, plan, ws, wsb, aux);
        if (st != CREDIT_OK) break;
        if (cudaEventRecord(e1, nullptr) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
            cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess) {
            st = CREDIT_ERR_CUDA;
            break;
        }
        if (r > 0) t.push_back(1e3 * ms);
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (st == CREDIT_OK) *us = median_of(t);
    return st;
}

// Elements of one CTA's staged slice that let `cps` CTAs share an SM (the
// one-row-per-cluster kernel's budget for one staged operand).
int64_t staged_budget(int dev, credit_op_t op, credit_dtype_t dtype, int cps) {
    const int es = dtype == CREDIT_F32 ? 4 : 2;
    const DevInfo* d = device_info(dev);
    const void* fn = cluster_kernel(KernelKey{(int)op, (int)dtype, 0, true, 1});
    const KernelInfo* ki = d ? kernel_info(dev, fn, true) : nullptr;
    if (!ki) return 0;
    const int64_t vec = 16 / es;
    int64_t budget = std::min<int64_t>(tail_budget_bytes(*d, ki->static_smem, cps),
                                       ki->max_dyn_smem);
    if (op == CREDIT_PEARSON) budget = budget / 2 - 128;  // x and u, one pitch apart
    return budget / (vec * es) * vec;
}

// The L2-tail staging forms of cluster size P (staged elements per slice, and
// threads per CTA, 0 for the planner's choice): the staged lengths that let
// two, three and (where the four-CTA instantiation exists) four CTAs share an
// SM; half the three-CTA length -- a longer tail that each warp writes from
// a ring of its freed staged tiles, whose loads overlap the staging from the
// start (measured faster for the widest bf16 softmax rows); and, for
// LayerNorm with the 64-register instantiation, the length for ten CTAs per
// SM at 128 threads each: small CTAs, seven or eight resident per SM
// (measured faster there, slower for softmax).  Empty where the operator has
// no L2-tail form.
struct TailForm {
    int64_t staged;
    int threads;
};
std::vector<TailForm> tail_forms(int dev, credit_op_t op, int64_t cols, credit_dtype_t dtype,
                                 int pdt, int P) {
    std::vector<TailForm> out;
    const bool quad = quad_capable((int)op, dtype == CREDIT_F32 ? 4 : 2, pdt == CREDIT_BF16 ? 2 : 4);
    for (int cps : {2, 3, 4}) {
        // four CTAs per SM only where the four-CTA instantiation exists
        if (cps == 4 && !quad) continue;
        const int64_t h = tail_staged_for(dev, op, cols, dtype, P, cps);
        if (h > 0) out.push_back({h, 0});
    }
    const int64_t vec = dtype == CREDIT_F32 ? 4 : 8;
    const int64_t h3 = tail_staged_for(dev, op, cols, dtype, P, 3);
    const int64_t half = h3 / 2 / vec * vec;
    if (h3 > 0 && half >= vec) out.push_back({half, 0});
    if (quad && op == CREDIT_LAYERNORM) {
        const int64_t h10 = tail_staged_for(dev, op, cols, dtype, P, 10);
        if (h10 > 0) out.push_back({h10, 128});
    }
    return out;
}

// The local-work primitive (a candidate's per-CTA work replayed without
// DSMEM; CREDIT "D. Profitability and Candidate Selection" builds its model
// from primitives matched to the candidate): the one-CTA-per-row kernel at
// cluster size 1 -- no exchange -- on a calibration matrix whose rows are
// one staged budget wide, so that `cps` CTAs share an SM, and `tails` more budgets of L2 tail
// (0: fully staged; 1: half the row in the tail; 3: three quarters).  GB/s of
// one read and one write of the matrix.
credit_status_t local_rate(int dev, credit_op_t op, credit_dtype_t dtype, int pdt, int cps,
                           int tails, int runs, double* gbps, int P = 1,
                           double* c_eff = nullptr) {
    const int es = dtype == CREDIT_F32 ? 4 : 2;
    const int64_t held = staged_budget(dev, op, dtype, cps);
    if (held < 16 / es) return CREDIT_ERR_NO_LEGAL_PLAN;
    const bool tail = tails > 0;
    const int64_t cols = held * (1 + tails) * P;
    const DevInfo* d = device_info(dev);
    if (!d) return CREDIT_ERR_CUDA;
    const int64_t row_bytes = cols * es;
    const int64_t rows = std::max<int64_t>((int64_t)8 * cps * d->sms,
                                           ceil_div64((int64_t)256 << 20, row_bytes));
    credit_plan_t p;
    credit_status_t st = make_plan(dev, op, rows, cols, dtype, CREDIT_CLUSTER, P, 0, 0, &p, 0, 1,
                                   tail ? held : 0);
    if (st != CREDIT_OK) return st;
    if (p.slice_elems != held * (1 + tails)) return CREDIT_ERR_NO_LEGAL_PLAN;
    if (c_eff) *c_eff = (double)p.active_clusters * P / (double)d->sms;
    {
        // a residency the footprint allows but threads or registers do not:
        // not a level of this primitive
        KernelKey key{(int)op, (int)dtype, pdt == CREDIT_BF16 ? 1 : 0, true, 1};
        key.deep = deep_footprint(dev, key, p.smem_bytes);
        key.quad = quad_footprint(dev, key, p.smem_bytes, p.staged_elems < p.slice_elems);
        const void* fn = cluster_kernel(key);
        int per_sm = 0;
        // kernel_info raises the instantiation's dynamic-SMEM limit first
        // (the occupancy calculator counts zero blocks otherwise)
        if (!fn || !kernel_info(dev, fn, true) ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, p.threads,
                                                          (size_t)p.smem_bytes) != cudaSuccess) {
            cudaGetLastError();
            return CREDIT_ERR_CUDA;
        }
        if (per_sm < cps) return CREDIT_ERR_NO_LEGAL_PLAN;
    }
    const bool pearson = op == CREDIT_PEARSON;
    const size_t mat = (size_t)rows * (size_t)row_bytes;
    const size_t pbytes = (size_t)cols * (pdt == CREDIT_F32 ? 4 : 2);
    Scratch x, y, g, b, aux;
    if (!x.alloc(mat) || !y.alloc(mat) || !aux.alloc((size_t)rows * 4) ||
        (pearson && !g.alloc(mat)) || (!pearson && pdt >= 0 && (!g.alloc(pbytes) || !b.alloc(pbytes))))
        return CREDIT_ERR_CUDA;
    const credit_dtype_t pd = pdt == CREDIT_BF16 ? CREDIT_BF16 : CREDIT_F32;
    if (!fill(x.p, rows * cols, dtype, -2.f, 2.f, 11u) ||
        (pearson && !fill(g.p, rows * cols, dtype, -2.f, 2.f, 12u)) ||
        (!pearson && pdt >= 0 &&
         (!fill(g.p, cols, pd, 0.5f, 1.5f, 13u) || !fill(b.p, cols, pd, -0.5f, 0.5f, 14u))) ||
        cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return CREDIT_ERR_CUDA;
    }
    double us = 0.0;
    st = time_op(op, x.p, y.p, rows, cols, dtype, g.p, b.p, pdt, &p, nullptr, 0, runs, &us,
                 static_cast<float*>(aux.p));
    if (st != CREDIT_OK) return st;
    const double bytes = (pearson ? 3.0 : (op == CREDIT_QUANTIZE ? 1.0 + 1.0 / es : 2.0)) * (double)mat;
    *gbps = bytes / us / 1e3;
    return CREDIT_OK;
}

double local_gbps(const LocalRates& r, double c_eff, double f);

// The primitive's rates of (op, dtype, pdt) at 1..4 CTAs per SM, measured once
// per device and kept (and persisted with the profile).
credit_status_t local_rates_for(int dev, credit_op_t op, credit_dtype_t dtype, int pdt, int runs,
                                LocalRates* out) {
    {
        std::lock_guard<std::mutex> lk(g_cm_mu);
        auto it = g_local.find(std::make_tuple(dev, (int)op, (int)dtype, pdt));
        if (it != g_local.end()) {
            *out = it->second;
            return CREDIT_OK;
        }
    }
    LocalRates r;
    std::memset(&r, 0, sizeof(r));
    r.op = (int)op;
    r.dtype = (int)dtype;
    r.pdt = pdt;
    const int es = dtype == CREDIT_F32 ? 4 : 2;
    const bool tails = tail_capable((int)op, es);
    for (int c = 1; c <= kLocalMaxCps; ++c) {
        credit_status_t st = local_rate(dev, op, dtype, pdt, c, 0, runs, &r.full[c]);
        if (st != CREDIT_OK && st != CREDIT_ERR_NO_LEGAL_PLAN) return st;
        if (st != CREDIT_OK) r.full[c] = 0.0;
        // the tail levels also where only L2-tail plans reach c CTAs per SM
        // (the four-CTA instantiation)
        if (st != CREDIT_OK && !quad_capable((int)op, es, pdt == CREDIT_BF16 ? 2 : 4)) continue;
        if (tails) {
            st = local_rate(dev, op, dtype, pdt, c, 1, runs, &r.tail50[c]);
            if (st != CREDIT_OK && st != CREDIT_ERR_NO_LEGAL_PLAN) return st;
            st = local_rate(dev, op, dtype, pdt, c, 3, runs, &r.tail75[c]);
            if (st != CREDIT_OK && st != CREDIT_ERR_NO_LEGAL_PLAN) return st;
        }
    }
    // the synchronisation factor of each cluster size: the clustered kernel
    // on rows of P calibration slices (three CTAs per SM) against the local
    // rate at the effective residency its clusters reach
    for (int P = 2; P <= kMaxCluster; ++P) {
        double g = 0.0, ce = 0.0;
        const credit_status_t st = local_rate(dev, op, dtype, pdt, 3, 0, runs, &g, P, &ce);
        if (st == CREDIT_ERR_NO_LEGAL_PLAN) continue;
        if (st != CREDIT_OK) return st;
        const double ref = local_gbps(r, ce, 0.0);
        if (ref > 0.0) r.sync[P] = std::min(1.0, g / ref);
    }
    local_rates_put(dev, r);
    *out = r;
    return CREDIT_OK;
}

// The primitive's rate at one whole residency c and L2-tail fraction f of
// the slice: piecewise linear in f through the fully staged rate and the
// rates with half and three quarters of the row in the tail, continued along
// the last piece beyond three quarters (floored at a tenth of the staged
// rate).
double local_gbps_at(const LocalRates& r, int c, double f) {
    const double full = r.full[c];
    if (full <= 0.0) {
        // a residency only L2-tail plans reach: flat below half the slice in
        // the tail, then along the tail levels
        if (r.tail50[c] <= 0.0) return 0.0;
        if (f <= 0.5) return r.tail50[c];
        const double t75 = r.tail75[c] > 0.0 ? r.tail75[c] : r.tail50[c];
        return std::max(0.1 * r.tail50[c], r.tail50[c] + (t75 - r.tail50[c]) * ((f - 0.5) / 0.25));
    }
    if (f <= 0.0 || r.tail50[c] <= 0.0) return full;
    if (f <= 0.5) return full + (r.tail50[c] - full) * (f / 0.5);
    const double t75 = r.tail75[c] > 0.0 ? r.tail75[c] : r.tail50[c];
    return std::max(0.1 * full, r.tail50[c] + (t75 - r.tail50[c]) * ((f - 0.5) / 0.25));
}

// ... at an effective residency c_eff (resident CTAs per SM, fractional):
// linear between the measured residencies around it (for a tail plan, also
// those only tail plans reach), proportional below one CTA per SM (idle SMs
// stream nothing), saturated at the highest residency measured.
double local_gbps(const LocalRates& r, double c_eff, double f) {
    if (r.full[1] <= 0.0) return 0.0;
    if (c_eff <= 1.0) return local_gbps_at(r, 1, f) * std::max(0.0, c_eff);
    int lo = 1;
    for (int c = 2; c <= kLocalMaxCps; ++c) {
        if (r.full[c] <= 0.0 && (f <= 0.0 || r.tail50[c] <= 0.0)) continue;
        if (c >= c_eff) {
            const double w = (c_eff - lo) / (double)(c - lo);
            return local_gbps_at(r, lo, f) * (1.0 - w) + local_gbps_at(r, c, f) * w;
        }
        lo = c;
    }
    return local_gbps_at(r, lo, f);
}

}  // namespace

extern "C" credit_status_t credit_plan_profiled(credit_op_t op, int64_t rows, int64_t cols,
                                                credit_dtype_t dtype, int param_dtype, int device,
                                                int runs, int tune, credit_plan_t* out,
                                                credit_model_report_t* report) {
    if (!out || rows < 1 || cols < 1 || runs < 1 || tune < 0 || device < 0 ||
        device >= kMaxDevices)
        return CREDIT_ERR_INVALID_ARG;
    if (dtype != CREDIT_F32 && dtype != CREDIT_BF16) return CREDIT_ERR_UNSUPPORTED;
    if (param_dtype != -1 && param_dtype != CREDIT_F32 && param_dtype != CREDIT_BF16)
        return CREDIT_ERR_UNSUPPORTED;
    profile_env_load(device);  // CREDIT_PROFILE: a saved DSMEM profile spares the calibration
    DsmemProfile prof;
    {
        std::lock_guard<std::mutex> lk(g_cm_mu);
        prof = g_profile[device];
    }
    if (!prof.valid) {
        const credit_status_t st = credit_calibrate(device, 7, nullptr);
        if (st != CREDIT_OK) return st;
        std::lock_guard<std::mutex> lk(g_cm_mu);
        prof = g_profile[device];
    }
    int old = 0;
    if (cudaGetDevice(&old) != cudaSuccess || cudaSetDevice(device) != cudaSuccess) {
        cudaGetLastError();
        return CREDIT_ERR_CUDA;
    }
    struct Restore { int d; ~Restore() { cudaSetDevice(d); } } restore{old};

    const DevInfo* d = device_info(device);
    if (!d) return CREDIT_ERR_CUDA;
    const int es = dtype == CREDIT_F32 ? 4 : 2;
    // the model times the shape's first `rt` rows: all of them up to 1 GiB of
    // input, so that scratch stays small next to a large resident workload
    const int64_t rt = std::max<int64_t>(1, std::min<int64_t>(rows, ((int64_t)1 << 30) / (cols * es)));
    const double mat = (double)rt * (double)cols * es;

    // the baseline: the fastest of local staging (when one CTA can hold a
    // row), one warp per row in registers (rows of at most 4 KiB) and the
    // two-pass re-read pair
    credit_plan_t base;
    const int64_t row_bytes = cols * es;
    const int Rb = row_bytes * 4 <= 65536 ? 4 : 1;
    credit_status_t st =
        make_plan(device, op, rt, cols, dtype, CREDIT_CLUSTER, 1, 0, 0, &base, 0, Rb);
    if (st != CREDIT_OK && Rb != 1)
        st = make_plan(device, op, rt, cols, dtype, CREDIT_CLUSTER, 1, 0, 0, &base, 0, 1);
    bool staging = st == CREDIT_OK;
    credit_plan_t reread;
    st = make_plan(device, op, rt, cols, dtype, CREDIT_TWO_PASS, 0, 0, 0, &reread);
    if (st != CREDIT_OK) return st;
    if (!staging) base = reread;
    // bytes: one read of x (and of u for Pearson) and one write of the
    // output (int8 codes for quantization); the re-read baseline reads the
    // inputs twice
    const bool pearson = op == CREDIT_PEARSON;
    const double b_read = pearson ? 2.0 * mat : mat;
    const double b_write = op == CREDIT_QUANTIZE ? (double)rt * (double)cols : mat;
    const double b_credit = b_read + b_write;

    // scratch buffers of the shape
    Scratch x, y, g, b, ws, aux;
    const size_t pbytes = (size_t)cols * (param_dtype == CREDIT_F32 ? 4 : 2);
    if (op == CREDIT_WEIGHTED_STD && param_dtype < 0) return CREDIT_ERR_INVALID_ARG;
    if (!x.alloc((size_t)mat) || !y.alloc((size_t)mat) || !aux.alloc((size_t)rt * 4) ||
        (pearson && !g.alloc((size_t)mat)) ||  // the second operand u
        (!pearson && param_dtype >= 0 && (!g.alloc(pbytes) || !b.alloc(pbytes))))
        return CREDIT_ERR_CUDA;
    if (!ws.alloc((size_t)reread.workspace_bytes)) return CREDIT_ERR_CUDA;
    const int64_t nmat = rt * cols;
    const credit_dtype_t pdt = param_dtype == CREDIT_BF16 ? CREDIT_BF16 : CREDIT_F32;
    if (!fill(x.p, nmat, dtype, -2.f, 2.f, 1u) ||
        (pearson && !fill(g.p, nmat, dtype, -2.f, 2.f, 2u)) ||
        (!pearson && param_dtype >= 0 &&
         (!fill(g.p, cols, pdt, 0.5f, 1.5f, 3u) || !fill(b.p, cols, pdt, -0.5f, 0.5f, 4u))) ||
        cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return CREDIT_ERR_CUDA;
    }

    double t_base = 0.0;
    float* auxp = static_cast<float*>(aux.p);
    st = time_op(op, x.p, y.p, rt, cols, dtype, g.p, b.p, param_dtype, &base, ws.p,
                 (size_t)base.workspace_bytes, runs, &t_base, auxp);
    if (st != CREDIT_OK) return st;
    if (staging) {
        double t_rr = 0.0;
        st = time_op(op, x.p, y.p, rt, cols, dtype, g.p, b.p, param_dtype, &reread, ws.p,
                     (size_t)reread.workspace_bytes, runs, &t_rr, auxp);
        if (st != CREDIT_OK) return st;
        if (t_rr < t_base) {
            staging = false;
            base = reread;
            t_base = t_rr;
        }
    }
    credit_plan_t wrows;
    if (make_plan(device, op, rt, cols, dtype, CREDIT_WARP_ROWS, 1, 0, 0, &wrows) == CREDIT_OK) {
        double t_wr = 0.0;
        st = time_op(op, x.p, y.p, rt, cols, dtype, g.p, b.p, param_dtype, &wrows, nullptr, 0,
                     runs, &t_wr, auxp);
        if (st != CREDIT_OK) return st;
        if (t_wr < t_base) {
            staging = true;  // one read of the row: no re-read to avoid
            base = wrows;
            t_base = t_wr;
        }
    }
    const double b_base = staging ? b_credit : b_credit + b_read;

    // the baseline's control: its grid, footprint and barriers, no work
    double ctrl_base = 0.0;
    if (base.variant == CREDIT_WARP_ROWS) {
        // a grid of row-striding CTAs: one launch, no staging, no barrier
        st = credit_control_time(device, base.active_clusters, 1, base.threads, 0, 1, 0, runs,
                                 &ctrl_base);
    } else if (staging) {
        st = credit_control_time(device, ceil_div64(rt, base.rows_per_cluster), 1, base.threads,
                                 base.smem_bytes, 1, 2, runs, &ctrl_base);
    } else {
        const int64_t nch = ceil_div64(cols, base.slice_elems);
        double one = 0.0;
        st = credit_control_time(device, rt * nch, 1, base.threads, 0, 1, 2, runs, &one);
        ctrl_base = 2.0 * one;  // two launches
    }
    if (st != CREDIT_OK) return st;

    credit_model_report_t rep;
    std::memset(&rep, 0, sizeof(rep));
    rep.baseline_variant = base.variant;
    rep.t_base_us = t_base;
    rep.b_base_bytes = b_base;
    rep.b_credit_bytes = b_credit;
    rep.t_ctrl_base_us = ctrl_base;
    rep.cand[0].cluster_size = 1;
    rep.cand[0].legal = 1;
    rep.cand[0].plan = base;
    rep.cand[0].pred_us = t_base;

    // The candidates' local work, valued by the local-work primitive at each
    // candidate's effective residency and L2-tail fraction instead of at the
    // baseline's achieved rate: a clustered plan moves its bytes at the rate
    // of the CTAs per SM its clusters keep resident.
    LocalRates lr;
    st = local_rates_for(device, op, dtype, param_dtype, runs, &lr);
    if (st != CREDIT_OK) return st;
    const int pkey = param_dtype == CREDIT_BF16 ? 1 : 0;

    double best = t_base;
    int best_P = 1;
    credit_plan_t chosen = base;
    for (int P = 2; P <= kMaxCluster; ++P) {
        credit_candidate_t& c = rep.cand[P - 1];
        c.cluster_size = P;
        // the whole slice staged (where it fits) and the L2-tail plans
        // (tail_forms)
        std::vector<credit_plan_t> plans;
        credit_plan_t p;
        if (make_plan(device, op, rt, cols, dtype, CREDIT_CLUSTER, P, 0, 0, &p, 0, 1) == CREDIT_OK)
            plans.push_back(p);
        for (const TailForm& f : tail_forms(device, op, cols, dtype, param_dtype, P)) {
            if (make_plan(device, op, rt, cols, dtype, CREDIT_CLUSTER, P, f.threads, 0, &p, 0, 1,
                          f.staged) == CREDIT_OK)
                plans.push_back(p);
        }
        for (const credit_plan_t& q : plans) {
            if ((int64_t)(P - 1) * q.slice_elems >= cols) continue;  // an idle CTA
            // residency: CTAs per SM the footprint allows, free of clusters
            KernelKey key{(int)op, (int)dtype, pkey, true, 1};
            key.deep = deep_footprint(device, key, q.smem_bytes);
            key.quad = quad_footprint(device, key, q.smem_bytes, q.staged_elems < q.slice_elems);
            const void* fn = cluster_kernel(key);
            int per_sm = 0;
            if (!fn || !kernel_info(device, fn, true) ||
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, q.threads,
                                                              (size_t)q.smem_bytes) !=
                    cudaSuccess ||
                per_sm < 1) {
                cudaGetLastError();
                continue;
            }
            // the CTAs per SM the candidate's clusters actually keep
            // resident: at most what the footprint allows, fewer where
            // clusters (which live in one GPC) cannot fill every slot
            const double c_eff = std::min<double>(
                per_sm, (double)q.active_clusters * P / (double)d->sms);
            const double f = q.staged_elems < q.slice_elems
                                 ? (double)(q.slice_elems - q.staged_elems) / (double)q.slice_elems
                                 : 0.0;
            // the cluster's synchronisation factor (a cluster waits for its
            // slowest CTA at the exchange), measured per cluster size
            const double sync = lr.sync[P] > 0.0 ? lr.sync[P] : 1.0;
            const double rate = local_gbps(lr, c_eff, f) * sync * 1e3;  // bytes per us
            if (rate <= 0.0) continue;
            const double waves = (double)ceil_div64(rt, q.active_clusters);
            const double quant = waves * q.active_clusters / (double)rt;  // last-wave fill
            const double t_local = b_credit / rate * quant;
            // DSMEM control: the cluster launch with its two barriers per row
            // over the same grid without clusters
            double ctrl = 0.0, ctrl1 = 0.0;
            st = credit_control_time(device, rt, P, q.threads, q.smem_bytes, 1, 2, runs, &ctrl);
            if (st == CREDIT_ERR_NO_LEGAL_PLAN) continue;
            if (st != CREDIT_OK) return st;
            st = credit_control_time(device, rt * P, 1, q.threads, q.smem_bytes, 1, 0, runs, &ctrl1);
            if (st != CREDIT_OK && st != CREDIT_ERR_NO_LEGAL_PLAN) return st;
            // the control kernel already pays the exchange's barrier; the push
            // costs what the measured exchange adds to it (with st.async
            // deposits the exchange replaces that barrier on the critical path)
            const double xchg_ns = q.exchange == CREDIT_EXCHANGE_ASYNC ? prof.async_exchange_ns[P]
                                                                       : prof.exchange_ns[P];
            const double push_ns = std::max(0.0, xchg_ns - prof.barrier_ns[P]);
            const double t_ctrl = std::max(0.0, ctrl - ctrl1);
            const double t_comm = waves * push_ns * 1e-3;
            // local replay: every CTA folds the P partials from its own shared
            // memory, one slot read per peer
            const double t_replay = waves * P * prof.local_load_ns * 1e-3;
            const double pred = t_local + t_ctrl + t_comm + t_replay;
            if (!c.legal || pred < c.pred_us) {
                c.legal = 1;
                c.plan = q;
                c.t_ctrl_us = t_ctrl;
                c.t_comm_us = t_comm + t_replay;
                c.pred_us = pred;
                c.plan.pred_us = (float)pred;
                c.plan.pred_two_pass_us = (float)t_base;
            }
        }
        if (c.legal && c.pred_us < best) {
            best = c.pred_us;
            best_P = P;
            chosen = c.plan;
        }
    }
    rep.model_cluster_size = best_P;
    rep.profitable = best_P > 1;
    chosen.pred_us = (float)best;
    chosen.pred_two_pass_us = (float)t_base;

    // final tuning: time the `tune` best-predicted candidates (and the
    // persistent and pipelined kernels of the same P) and keep the fastest
    // measured plan
    if (tune > 0) {
        std::vector<int> order;
        for (int P = 2; P <= kMaxCluster; ++P)
            if (rep.cand[P - 1].legal) order.push_back(P);
        std::sort(order.begin(), order.end(), [&](int a2, int b2) {
            return rep.cand[a2 - 1].pred_us < rep.cand[b2 - 1].pred_us;
        });
        if ((int)order.size() > tune) order.resize(tune);
        double best_meas = t_base;
        credit_plan_t best_plan = base;
        int best_meas_P = 1;
        rep.cand[0].measured_us = t_base;
        // every timed clustered plan, for the confirmation round below
        struct Timed {
            double us;
            credit_plan_t plan;
            int P;
        };
        std::vector<Timed> timed;
        for (int P : order) {
            credit_candidate_t& c = rep.cand[P - 1];
            // the model's plan of this P, then its other staging forms: the
            // whole slice (where it fits) and the L2-tail plans (tail_forms)
            std::vector<credit_plan_t> plans{c.plan};
            credit_plan_t tp;
            if (c.plan.staged_elems < c.plan.slice_elems &&
                make_plan(device, op, rt, cols, dtype, CREDIT_CLUSTER, P, 0, 0, &tp, 0, 1) == CREDIT_OK)
                plans.push_back(tp);
            for (const TailForm& f : tail_forms(device, op, cols, dtype, param_dtype, P)) {
                if ((f.staged != c.plan.staged_elems ||
                     (f.threads != 0 && f.threads != c.plan.threads)) &&
                    make_plan(device, op, rt, cols, dtype, CREDIT_CLUSTER, P, f.threads, 0, &tp,
                              0, 1, f.staged) == CREDIT_OK)
                    plans.push_back(tp);
            }
            for (size_t i = 0; i < plans.size(); ++i) {
                double us = 0.0;
                st = time_op(op, x.p, y.p, rt, cols, dtype, g.p, b.p, param_dtype, &plans[i],
                             nullptr, 0, runs, &us, auxp);
                if (st != CREDIT_OK) return st;
                if (i == 0) c.measured_us = us;
                timed.push_back({us, plans[i], P});
                if (plans[i].staged_elems < plans[i].slice_elems &&
                    (c.tail_us == 0.0 || us < c.tail_us)) {
                    c.tail_us = us;
                    c.tail_staged_elems = plans[i].staged_elems;
                }
                if (us < best_meas) {
                    best_meas = us;
                    best_plan = plans[i];
                    best_meas_P = P;
                }
            }
            // operators with per-column parameters: two rows per cluster
            // share one parameter load; their L2-tail plans keep the CTAs
            // per SM of a one-row plan
            if ((op == CREDIT_LAYERNORM || op == CREDIT_RMSNORM) && param_dtype >= 0 && rt >= 2) {
                for (int cps : {2, 3}) {
                    const int64_t held = tail_staged_for(device, op, cols, dtype, P, cps, 2);
                    credit_plan_t rp;
                    if (held == 0 || make_plan(device, op, rt, cols, dtype, CREDIT_CLUSTER, P, 0,
                                               0, &rp, 0, 2, held) != CREDIT_OK)
                        continue;
                    double us = 0.0;
                    st = time_op(op, x.p, y.p, rt, cols, dtype, g.p, b.p, param_dtype, &rp,
                                 nullptr, 0, runs, &us, auxp);
                    if (st != CREDIT_OK) return st;
                    timed.push_back({us, rp, P});
                    if (c.tail_us == 0.0 || us < c.tail_us) {
                        c.tail_us = us;
                        c.tail_staged_elems = held;
                    }
                    if (us < best_meas) {
                        best_meas = us;
                        best_plan = rp;
                        best_meas_P = P;
                    }
                }
            }
            for (credit_variant_t rv : {CREDIT_CLUSTER_PERSISTENT, CREDIT_CLUSTER_PIPELINED}) {
                credit_plan_t pp;
                if (make_plan(device, op, rt, cols, dtype, rv, P, 0, 0, &pp) != CREDIT_OK) continue;
                double* us = rv == CREDIT_CLUSTER_PERSISTENT ? &c.persistent_us : &c.pipelined_us;
                st = time_op(op, x.p, y.p, rt, cols, dtype, g.p, b.p, param_dtype, &pp, nullptr,
                             0, runs, us, auxp);
                if (st != CREDIT_OK) return st;
                timed.push_back({*us, pp, P});
                if (*us < best_meas) {
                    best_meas = *us;
                    best_plan = pp;
                    best_meas_P = P;
                }
            }
        }
        // confirmation: the three fastest timed plans are timed twice more,
        // interleaved, and ranked by the mean of their three medians, so that
        // one noisy median cannot decide between candidates a percent apart
        std::sort(timed.begin(), timed.end(),
                  [](const Timed& a, const Timed& b) { return a.us < b.us; });
        const size_t nk = std::min<size_t>(3, timed.size());
        if (nk > 1) {
            std::vector<double> sum(nk);
            for (size_t i = 0; i < nk; ++i) sum[i] = timed[i].us;
            for (int round = 0; round < 2; ++round) {
                for (size_t i = 0; i < nk; ++i) {
                    double us = 0.0;
                    st = time_op(op, x.p, y.p, rt, cols, dtype, g.p, b.p, param_dtype,
                                 &timed[i].plan, nullptr, 0, runs, &us, auxp);
                    if (st != CREDIT_OK) return st;
                    sum[i] += us;
                }
            }
            size_t bi = 0;
            for (size_t i = 1; i < nk; ++i)
                if (sum[i] < sum[bi]) bi = i;
            if (sum[bi] / 3.0 < t_base) {
                best_meas = sum[bi] / 3.0;
                best_plan = timed[bi].plan;
                best_meas_P = timed[bi].P;
            } else {
                best_meas = t_base;
                best_plan = base;
                best_meas_P = 1;
            }
        }
        chosen = best_plan;
        chosen.pred_us = (float)best_meas;
        chosen.pred_two_pass_us = (float)t_base;
        best_P = best_meas_P;
    }
    rep.chosen_cluster_size = best_P;
    rep.chosen_variant = chosen.variant;
    if (rt != rows) {
        // the chosen configuration, planned for every row of the shape
        credit_plan_t full;
        const credit_variant_t v = (credit_variant_t)chosen.variant;
        const bool pers = v == CREDIT_CLUSTER_PERSISTENT || v == CREDIT_CLUSTER_PIPELINED;
        if (make_plan(device, op, rows, cols, dtype, v, chosen.cluster_size, chosen.threads,
                      pers ? chosen.ctas_per_sm : 0, &full, pers ? chosen.chunk_elems : 0,
                      v == CREDIT_CLUSTER ? chosen.rows_per_cluster : 0,
                      v == CREDIT_CLUSTER ? chosen.staged_elems : 0) == CREDIT_OK) {
            const double scale = (double)rows / (double)rt;
            full.exchange = chosen.exchange;
            full.pred_us = (float)(chosen.pred_us * scale);
            full.pred_two_pass_us = (float)(chosen.pred_two_pass_us * scale);
            chosen = full;
        }
    }
    {
        std::lock_guard<std::mutex> lk(g_cm_mu);
        g_chosen[std::make_tuple(device, (int)op, (int)dtype, rows, cols)] = chosen;
    }
    profile_env_save(device);
    *out = chosen;
    if (report) *report = rep;
    return CREDIT_OK;
}
