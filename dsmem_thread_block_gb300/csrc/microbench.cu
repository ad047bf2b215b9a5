// microbench.cu -- DSMEM primitive characterisation and the control kernel.
//
// CREDIT summary page (arXiv 2609.01864v1), "C. Positioning": DSMEM is
// characterised by latency, throughput and repeated cluster-barrier
// benchmarks whose CTAs sit on different SMs, each reported as the median of
// 15 runs.  "D. Profitability and Candidate Selection": a control kernel that
// does no work but copies the real kernel's grid, cluster size,
// shared-memory footprint and two barriers per row measures what launching,
// scheduling, occupancy and synchronisation cost; T_ctrl is its time beyond
// a control without clusters.
//
// Every benchmark kernel requests more than half of an SM's shared memory
// (or the caller's footprint) so that no two of its CTAs share an SM; the
// SM ids are reported so the caller can check.  Timing inside kernels uses
// clock64 (SM cycles) and %globaltimer (ns); the control kernel is timed
// with CUDA events.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <vector>

#include "credit.h"
#include "common.cuh"
#include "internal.h"
#include "planner.h"

namespace credit {
namespace {

struct BenchOut {
    long long cycles;     // measured by rank 0, thread 0
    long long ns;
    unsigned smid[kMaxCluster];
    unsigned sink;
    unsigned err;         // a bounded wait gave up
};

constexpr uint64_t kBenchWaitNs = 100000000ull;  // 0.1 s per exchange wait

constexpr int kChaseEntries = 4096;      // u32 ring in shared memory
constexpr int kBwBytes = 64 * 1024;      // remote buffer for the throughput kinds

__device__ __forceinline__ void cluster_sync_all() {
    cluster_arrive_release();
    cluster_wait_acquire();
}

// kind BARRIER: iters x (arrive.release + wait.acquire) on a cluster of P.
// kind EXCHANGE: iters x (push a 16-byte partial to every peer + barrier),
// i.e. steps a4 + a5 of the protocol.
__global__ void bench_barrier(BenchOut* out, int iters, int exchange) {
    __shared__ __align__(16) float slots[kMaxCluster * 4];
    const uint32_t P = cluster_nctarank(), rank = cluster_ctarank();
    if (threadIdx.x == 0) out->smid[rank] = smid();
    cluster_sync_all();
    const long long c0 = clock64();
    const uint64_t t0 = globaltimer_ns();
    for (int i = 0; i < iters; ++i) {
        if (exchange && threadIdx.x < P) {
            const uint32_t dst = mapa_shared(smem_u32(&slots[rank * 4]), threadIdx.x);
            st_cluster_v4f32(dst, (float)i, 1.f, 2.f, 3.f);
        }
        cluster_sync_all();
    }
    const long long c1 = clock64();
    const uint64_t t1 = globaltimer_ns();
    if (rank == 0 && threadIdx.x == 0) {
        out->cycles = c1 - c0;
        out->ns = (long long)(t1 - t0);
        out->sink = (unsigned)slots[0];
    }
    cluster_sync_all();
}

// kind ASYNC_EXCHANGE: iters x (st.async of a 16-byte partial into every
// peer, counted on the peer's mbarrier, then a wait on the CTA's own
// mbarrier for its P - 1 deposits) -- the exchange without a cluster barrier.
// Two mbarriers and two slot arrays alternate by iteration: a peer can be at
// most one exchange ahead (its next wait needs this CTA's next deposit), so
// a deposit never lands in the phase or the slots of the exchange before.
__global__ void bench_async_exchange(BenchOut* out, int iters) {
    __shared__ __align__(16) float slots[2][kMaxCluster * 4];
    __shared__ __align__(8) uint64_t bar[2];
    const uint32_t P = cluster_nctarank(), rank = cluster_ctarank();
    const uint32_t bytes = (P - 1) * 16u;
    if (threadIdx.x == 0) {
        out->smid[rank] = smid();
        mbar_init(smem_u32(&bar[0]), 1);
        mbar_init(smem_u32(&bar[1]), 1);
        fence_mbar_init();
    }
    cluster_sync_all();
    const long long c0 = clock64();
    const uint64_t t0 = globaltimer_ns();
    // warp 0 alone exchanges; the warp-wide vote after each wait keeps its
    // lanes within one phase of each other (no lane can miss a phase of the
    // mbarrier it waits on) and makes a give-up uniform across the warp
    for (int i = 0; threadIdx.x < 32 && i < iters; ++i) {
        const int b = i & 1;
        const uint32_t lb = smem_u32(&bar[b]);
        if (threadIdx.x == 0) mbar_arrive_expect_tx(lb, bytes);
        if (threadIdx.x < P && threadIdx.x != rank) {
            const uint32_t dst = mapa_shared(smem_u32(&slots[b][rank * 4]), threadIdx.x);
            st_async_v4f32(dst, (float)i, 1.f, 2.f, 3.f, mapa_shared(lb, threadIdx.x));
        }
        const bool ok = mbar_wait_limited(lb, (uint32_t)(i >> 1) & 1u, &out->err, kBenchWaitNs);
        if (!__all_sync(0xffffffffu, ok)) break;
    }
    const long long c1 = clock64();
    const uint64_t t1 = globaltimer_ns();
    if (rank == 0 && threadIdx.x == 0) {
        out->cycles = c1 - c0;
        out->ns = (long long)(t1 - t0);
        out->sink = (unsigned)slots[0][4 * (P - 1)];
    }
    cluster_sync_all();  // every deposit has landed before any CTA exits
}

// kind LOAD_LATENCY: rank 0 chases a pointer ring that lives in rank 1's
// shared memory (remote) or in its own (local).
__global__ void bench_chase(BenchOut* out, int iters, int remote) {
    __shared__ uint32_t ring[kChaseEntries];
    const uint32_t rank = cluster_ctarank();
    if (threadIdx.x == 0) out->smid[rank] = smid();
    // a stride coprime with the ring size defeats any prefetch
    for (int i = threadIdx.x; i < kChaseEntries; i += blockDim.x)
        ring[i] = (uint32_t)((i + 1031) % kChaseEntries);
    __syncthreads();
    cluster_sync_all();
    if (rank == 0 && threadIdx.x == 0) {
        const uint32_t owner = remote ? 1u : 0u;
        const uint32_t base = mapa_shared(smem_u32(ring), owner);
        uint32_t idx = 0;
        const long long c0 = clock64();
        const uint64_t t0 = globaltimer_ns();
        for (int i = 0; i < iters; ++i) idx = ld_cluster_u32(base + idx * 4u);
        const long long c1 = clock64();
        const uint64_t t1 = globaltimer_ns();
        out->cycles = c1 - c0;
        out->ns = (long long)(t1 - t0);
        out->sink = idx;
    }
    cluster_sync_all();  // rank 1 keeps its shared memory alive until rank 0 is done
}

// kind STORE_BW / LOAD_BW: every thread of rank 0 moves 16-byte vectors to or
// from a 64 KiB buffer of rank 1 (remote) or of its own (local), `iters`
// passes over the buffer.
__global__ void bench_bw(BenchOut* out, int iters, int remote, int store) {
    extern __shared__ __align__(16) unsigned char buf[];
    const uint32_t rank = cluster_ctarank();
    if (threadIdx.x == 0) out->smid[rank] = smid();
    for (int i = threadIdx.x; i < kBwBytes / 4; i += blockDim.x)
        reinterpret_cast<uint32_t*>(buf)[i] = (uint32_t)i;
    __syncthreads();
    cluster_sync_all();
    if (rank == 0) {
        const uint32_t base = mapa_shared(smem_u32(buf), remote ? 1u : 0u);
        uint32_t acc = 0;
        __syncthreads();
        const long long c0 = clock64();
        const uint64_t t0 = globaltimer_ns();
        for (int it = 0; it < iters; ++it) {
            for (int v = threadIdx.x; v < kBwBytes / 16; v += blockDim.x) {
                const uint32_t addr = base + (uint32_t)v * 16u;
                if (store) {
                    st_cluster_v4f32(addr, (float)it, (float)v, 0.f, 1.f);
                } else {
                    uint32_t a0, a1, a2, a3;
                    asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3) : "r"(addr) : "memory");
                    acc ^= a0 ^ a1 ^ a2 ^ a3;
                }
            }
        }
        if (store) asm volatile("fence.acq_rel.cluster;" ::: "memory");
        __syncthreads();
        const long long c1 = clock64();
        const uint64_t t1 = globaltimer_ns();
        if (threadIdx.x == 0) {
            out->cycles = c1 - c0;
            out->ns = (long long)(t1 - t0);
        }
        if (acc == 0xdeadbeefu) out->sink = acc;
    }
    cluster_sync_all();
}

// The control kernel: the real kernel's grid (nclusters x P CTAs), cluster
// size, dynamic shared memory and `barriers` cluster barriers per row for
// `rows_per_cluster` rows, and no work.
// The dynamic shared memory is only requested at launch (it sets residency);
// the kernel never touches it, so a zero-byte footprint is valid too.
__global__ void control_kernel(int rows_per_cluster, int barriers) {
    const bool clustered = cluster_nctarank() > 1;
    for (int r = 0; r < rows_per_cluster; ++r)
        for (int b = 0; b < barriers; ++b)
            if (clustered) cluster_sync_all();
            else __syncthreads();
}

// The staged-copy primitive: every CTA moves one footprint of bytes HBM ->
// shared memory (non-multicast bulk copies, one mbarrier per 16 KiB chunk),
// reads it back once chunk by chunk as it lands (a fold standing in for the
// statistics pass), meets at a block barrier (the partial), then reads it a
// second time and stores it to HBM (streaming 16-byte stores): the data
// movement and shared-memory passes of a one-pass reduce-reuse CTA without
// its arithmetic or exchange.  The footprint sets how many CTAs share an SM,
// so its rate at k CTAs per SM is the measured streaming rate of that
// residency.
constexpr int kStageChunk = 16384;
__global__ void __launch_bounds__(256) stage_copy_kernel(const unsigned char* src,
                                                         unsigned char* dst, int footprint,
                                                         unsigned* err) {
    extern __shared__ __align__(128) unsigned char stage_buf[];
    __shared__ __align__(8) uint64_t bar[kMaxChunks];
    unsigned char* buf = stage_buf;
    const int nch = footprint / kStageChunk;
    const int64_t base = (int64_t)blockIdx.x * footprint;
    if (threadIdx.x == 0) {
        for (int c = 0; c < nch; ++c) mbar_init(smem_u32(&bar[c]), 1);
        fence_mbar_init();
        fence_proxy_async_smem();
        const uint64_t pol = l2_policy_evict_first();
        for (int c = 0; c < nch; ++c) {
            const uint32_t b = smem_u32(&bar[c]);
            mbar_arrive_expect_tx(b, (uint32_t)kStageChunk);
            bulk_g2s(smem_u32(buf) + (uint32_t)(c * kStageChunk), src + base + (int64_t)c * kStageChunk,
                     (uint32_t)kStageChunk, b, pol);
        }
    }
    __syncthreads();
    uint32_t fold = 0;
    for (int c = 0; c < nch; ++c) {
        mbar_wait_bounded(smem_u32(&bar[c]), 0, err);
        const unsigned char* s = buf + c * kStageChunk;
        for (int v = threadIdx.x; v < kStageChunk / 16; v += blockDim.x) {
            const uint4 q = lds16(s + v * 16);
            fold += q.x ^ q.y ^ q.z ^ q.w;
        }
    }
    // keeps the fold live (footprint is never negative, which the compiler
    // cannot know)
    if (footprint < 0) err[1] = fold;
    __syncthreads();
    for (int c = 0; c < nch; ++c) {
        const unsigned char* s = buf + c * kStageChunk;
        unsigned char* d = dst + base + (int64_t)c * kStageChunk;
        for (int v = threadIdx.x; v < kStageChunk / 16; v += blockDim.x)
            stg16_stream(d + (int64_t)v * 16, lds16(s + v * 16));
    }
}

cudaError_t launch_cluster_kernel(const void* fn, int P, int ctas, int threads, size_t smem,
                                  void** args, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas, 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)P;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = P > 1 ? 1 : 0;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

double median(std::vector<double> v) {
    std::sort(v.begin(), v.end());
    const size_t n = v.size();
    return n % 2 ? v[n / 2] : 0.5 * (v[n / 2 - 1] + v[n / 2]);
}

double quantile(std::vector<double> v, double q) {
    std::sort(v.begin(), v.end());
    const double pos = q * (double)(v.size() - 1);
    const size_t i = (size_t)pos;
    const double f = pos - (double)i;
    return i + 1 < v.size() ? v[i] * (1 - f) + v[i + 1] * f : v[i];
}

}  // namespace
}  // namespace credit

using namespace credit;

extern "C" credit_status_t credit_bench_dsmem(int device, int kind, int cluster_size, int iters,
                                              int runs, credit_bench_result_t* out) {
    if (!out || iters < 1 || runs < 1 || runs > 1000) return CREDIT_ERR_INVALID_ARG;
    if (cluster_size < 1 || cluster_size > kMaxCluster) return CREDIT_ERR_INVALID_ARG;
    const bool pair = kind == CREDIT_BENCH_REMOTE_LOAD_LATENCY || kind == CREDIT_BENCH_LOCAL_LOAD_LATENCY ||
                      kind == CREDIT_BENCH_REMOTE_STORE_BW || kind == CREDIT_BENCH_REMOTE_LOAD_BW ||
                      kind == CREDIT_BENCH_LOCAL_STORE_BW || kind == CREDIT_BENCH_LOCAL_LOAD_BW;
    if (!pair && kind != CREDIT_BENCH_BARRIER && kind != CREDIT_BENCH_EXCHANGE &&
        kind != CREDIT_BENCH_ASYNC_EXCHANGE)
        return CREDIT_ERR_INVALID_ARG;
    const int P = pair ? 2 : cluster_size;
    const DevInfo* d = device_info(device);
    if (!d) return CREDIT_ERR_CUDA;
    int old = 0;
    if (cudaGetDevice(&old) != cudaSuccess || cudaSetDevice(device) != cudaSuccess) {
        cudaGetLastError();
        return CREDIT_ERR_CUDA;
    }
    credit_status_t status = CREDIT_OK;
    BenchOut* dout = nullptr;
    std::vector<double> cyc, ns;
    BenchOut h;
    std::memset(&h, 0, sizeof(h));
    const void* fn = nullptr;
    int threads = 32;
    size_t smem = (size_t)d->smem_per_sm / 2 + 4096;  // one CTA per SM
    int remote = (kind == CREDIT_BENCH_REMOTE_LOAD_LATENCY || kind == CREDIT_BENCH_REMOTE_STORE_BW ||
                  kind == CREDIT_BENCH_REMOTE_LOAD_BW);
    int store = (kind == CREDIT_BENCH_REMOTE_STORE_BW || kind == CREDIT_BENCH_LOCAL_STORE_BW);
    int exchange = kind == CREDIT_BENCH_EXCHANGE;
    if (kind == CREDIT_BENCH_BARRIER || kind == CREDIT_BENCH_EXCHANGE) {
        fn = (const void*)bench_barrier;
        threads = 128;
    } else if (kind == CREDIT_BENCH_ASYNC_EXCHANGE) {
        fn = (const void*)bench_async_exchange;
        threads = 128;
    } else if (kind == CREDIT_BENCH_REMOTE_LOAD_LATENCY || kind == CREDIT_BENCH_LOCAL_LOAD_LATENCY) {
        fn = (const void*)bench_chase;
        threads = 128;
    } else {
        fn = (const void*)bench_bw;
        threads = 512;
        smem = std::max<size_t>(smem, kBwBytes);
    }
    if (!kernel_info(device, fn, true)) status = CREDIT_ERR_CUDA;
    if (status == CREDIT_OK && cudaMalloc(&dout, sizeof(BenchOut)) != cudaSuccess) status = CREDIT_ERR_CUDA;
    for (int r = 0; status == CREDIT_OK && r < runs + 1; ++r) {  // run 0 warms up
        void* args_barrier[] = {&dout, &iters, &exchange};
        void* args_chase[] = {&dout, &iters, &remote};
        void* args_bw[] = {&dout, &iters, &remote, &store};
        void* args_async[] = {&dout, &iters};
        void** args = fn == (const void*)bench_barrier ? args_barrier
                      : fn == (const void*)bench_chase ? args_chase
                      : fn == (const void*)bench_async_exchange ? args_async : args_bw;
        if (cudaMemset(dout, 0, sizeof(BenchOut)) != cudaSuccess ||
            launch_cluster_kernel(fn, P, P, threads, smem, args, 0) != cudaSuccess ||
            cudaDeviceSynchronize() != cudaSuccess ||
            cudaMemcpy(&h, dout, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) {
            cudaGetLastError();
            status = CREDIT_ERR_CUDA;
            break;
        }
        if (h.err) {
            status = CREDIT_ERR_DEVICE_TIMEOUT;
            break;
        }
        if (r == 0) continue;
        cyc.push_back((double)h.cycles / iters);
        ns.push_back((double)h.ns / iters);
    }
    if (dout) cudaFree(dout);
    cudaSetDevice(old);
    if (status != CREDIT_OK) return status;
    std::memset(out, 0, sizeof(*out));
    out->kind = kind;
    out->cluster_size = P;
    out->runs = runs;
    for (int q = 0; q < P; ++q) out->smids[q] = (int32_t)h.smid[q];
    out->median_cycles = median(cyc);
    out->median_ns = median(ns);
    out->iqr_cycles = quantile(cyc, 0.75) - quantile(cyc, 0.25);
    if (pair && kind != CREDIT_BENCH_REMOTE_LOAD_LATENCY && kind != CREDIT_BENCH_LOCAL_LOAD_LATENCY) {
        out->bytes_per_cycle = (double)kBwBytes / out->median_cycles;
        out->gbps = (double)kBwBytes / out->median_ns;
    }
    return CREDIT_OK;
}

extern "C" credit_status_t credit_control_time(int device, int64_t nclusters, int cluster_size,
                                               int threads, int64_t smem_bytes,
                                               int rows_per_cluster, int barriers_per_row,
                                               int runs, double* median_us) {
    if (!median_us || nclusters < 1 || nclusters * cluster_size > 0x7fffffff || runs < 1 ||
        cluster_size < 1 || cluster_size > kMaxCluster || threads < 32 || threads > 1024 ||
        smem_bytes < 0 || rows_per_cluster < 0 || barriers_per_row < 0)
        return CREDIT_ERR_INVALID_ARG;
    const DevInfo* d = device_info(device);
    if (!d) return CREDIT_ERR_CUDA;
    const KernelInfo* ki = kernel_info(device, (const void*)control_kernel, true);
    if (!ki) return CREDIT_ERR_CUDA;
    if (smem_bytes > ki->max_dyn_smem) return CREDIT_ERR_NO_LEGAL_PLAN;
    int old = 0;
    if (cudaGetDevice(&old) != cudaSuccess || cudaSetDevice(device) != cudaSuccess) {
        cudaGetLastError();
        return CREDIT_ERR_CUDA;
    }
    credit_status_t status = CREDIT_OK;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    std::vector<double> t;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) status = CREDIT_ERR_CUDA;
    for (int r = 0; status == CREDIT_OK && r < runs + 1; ++r) {
        void* args[] = {&rows_per_cluster, &barriers_per_row};
        float ms = 0.f;
        if (cudaEventRecord(e0, 0) != cudaSuccess ||
            launch_cluster_kernel((const void*)control_kernel, cluster_size,
                                  (int)(nclusters * cluster_size), threads, (size_t)smem_bytes, args,
                                  0) != cudaSuccess ||
            cudaEventRecord(e1, 0) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
            cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess) {
            cudaGetLastError();
            status = CREDIT_ERR_CUDA;
            break;
        }
        if (r > 0) t.push_back(1e3 * ms);
    }
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    cudaSetDevice(old);
    if (status == CREDIT_OK) *median_us = median(t);
    return status;
}

// L2 read primitive: every CTA reads the whole `window` (16-byte vectors,
// eight loads in flight per thread, past L1), starting at a CTA-dependent
// offset so the CTAs spread over the L2 slices.  With a window far smaller
// than L2 every read after the first launch is an L2 hit: the rate is what
// the SMs can pull from L2 at once -- the ceiling of a stream that re-reads
// the same per-column vectors row after row.
__global__ void __launch_bounds__(512) l2_read_kernel(const uint4* window, int64_t nvec,
                                                      unsigned* sink) {
    constexpr int U = 8;
    const int64_t start = ((int64_t)blockIdx.x * 9973) % nvec;
    uint32_t fold = 0;
    for (int64_t i0 = threadIdx.x; i0 < nvec; i0 += (int64_t)U * blockDim.x) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            int64_t i = i0 + (int64_t)u * blockDim.x;
            if (i < nvec) {
                i += start;
                if (i >= nvec) i -= nvec;
                v[u] = ld_global_nc_l1na_v4(window + i);
            } else {
                v[u] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) fold += v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
    }
    // keeps the loads live (nvec is never negative, which the compiler
    // cannot know)
    if (nvec < 0) sink[0] = fold;
}

extern "C" credit_status_t credit_l2_read_rate(int device, int64_t window_bytes, int runs,
                                               double* gbps) {
    if (!gbps || window_bytes < 65536 || window_bytes > ((int64_t)64 << 20) || window_bytes % 16 ||
        runs < 1 || runs > 1000)
        return CREDIT_ERR_INVALID_ARG;
    const DevInfo* d = device_info(device);
    if (!d) return CREDIT_ERR_CUDA;
    const KernelInfo* ki = kernel_info(device, (const void*)l2_read_kernel, false);
    if (!ki) return CREDIT_ERR_CUDA;
    int old = 0;
    if (cudaGetDevice(&old) != cudaSuccess || cudaSetDevice(device) != cudaSuccess) {
        cudaGetLastError();
        return CREDIT_ERR_CUDA;
    }
    struct Restore { int d; ~Restore() { cudaSetDevice(d); } } restore{old};
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, l2_read_kernel, 512, 0) != cudaSuccess ||
        occ < 1) {
        cudaGetLastError();
        return CREDIT_ERR_CUDA;
    }
    const int64_t ctas = (int64_t)occ * d->sms;
    unsigned* err = device_error_word();
    if (!err) return CREDIT_ERR_CUDA;
    void* w = nullptr;
    if (cudaMalloc(&w, (size_t)window_bytes) != cudaSuccess ||
        cudaMemset(w, 0x5a, (size_t)window_bytes) != cudaSuccess) {
        cudaGetLastError();
        if (w) cudaFree(w);
        return CREDIT_ERR_CUDA;
    }
    const int64_t nvec = window_bytes / 16;
    credit_status_t status = CREDIT_OK;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    std::vector<double> t;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) status = CREDIT_ERR_CUDA;
    for (int r = 0; status == CREDIT_OK && r < runs + 1; ++r) {  // run 0 warms up (fills L2)
        float ms = 0.f;
        if (cudaEventRecord(e0, 0) != cudaSuccess) { status = CREDIT_ERR_CUDA; break; }
        l2_read_kernel<<<(unsigned)ctas, 512>>>(static_cast<const uint4*>(w), nvec, err);
        if (cudaGetLastError() != cudaSuccess || cudaEventRecord(e1, 0) != cudaSuccess ||
            cudaEventSynchronize(e1) != cudaSuccess || cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess) {
            cudaGetLastError();
            status = CREDIT_ERR_CUDA;
            break;
        }
        if (r > 0) t.push_back(1e3 * ms);
    }
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    cudaFree(w);
    if (status != CREDIT_OK) return status;
    *gbps = (double)ctas * (double)window_bytes / median(t) / 1e3;  // bytes / us / 1e3 = GB/s
    return CREDIT_OK;
}

extern "C" credit_status_t credit_stage_copy_rate(int device, int ctas_per_sm, int runs,
                                                  double* gbps, int* resident) {
    if (!gbps || ctas_per_sm < 1 || ctas_per_sm > 8 || runs < 1 || runs > 1000)
        return CREDIT_ERR_INVALID_ARG;
    const DevInfo* d = device_info(device);
    if (!d) return CREDIT_ERR_CUDA;
    const KernelInfo* ki = kernel_info(device, (const void*)stage_copy_kernel, false);
    if (!ki) return CREDIT_ERR_CUDA;
    // the largest whole number of 16 KiB chunks that lets ctas_per_sm CTAs
    // share an SM's shared memory
    const int64_t per_cta = (int64_t)d->smem_per_sm / ctas_per_sm - ki->static_smem - d->reserved_smem;
    int64_t fp = std::min<int64_t>(per_cta, ki->max_dyn_smem) / kStageChunk * kStageChunk;
    fp = std::min<int64_t>(fp, (int64_t)kMaxChunks * kStageChunk);
    if (fp < kStageChunk) return CREDIT_ERR_NO_LEGAL_PLAN;
    int old = 0;
    if (cudaGetDevice(&old) != cudaSuccess || cudaSetDevice(device) != cudaSuccess) {
        cudaGetLastError();
        return CREDIT_ERR_CUDA;
    }
    struct Restore { int d; ~Restore() { cudaSetDevice(d); } } restore{old};
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, stage_copy_kernel, 256, (size_t)fp) !=
        cudaSuccess) {
        cudaGetLastError();
        return CREDIT_ERR_CUDA;
    }
    if (resident) *resident = occ;
    const int64_t ctas = std::max<int64_t>((int64_t)4 * occ * d->sms, ((int64_t)512 << 20) / fp);
    const int64_t bytes = ctas * fp;
    unsigned* err = device_error_word();
    if (!err) return CREDIT_ERR_CUDA;
    void* src = nullptr;
    void* dst = nullptr;
    if (cudaMalloc(&src, (size_t)bytes) != cudaSuccess || cudaMalloc(&dst, (size_t)bytes) != cudaSuccess ||
        cudaMemset(src, 0, (size_t)bytes) != cudaSuccess) {
        cudaGetLastError();
        if (src) cudaFree(src);
        if (dst) cudaFree(dst);
        return CREDIT_ERR_CUDA;
    }
    credit_status_t status = CREDIT_OK;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    std::vector<double> t;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) status = CREDIT_ERR_CUDA;
    int fpi = (int)fp;
    const unsigned char* s = static_cast<const unsigned char*>(src);
    unsigned char* dd = static_cast<unsigned char*>(dst);
    for (int r = 0; status == CREDIT_OK && r < runs + 1; ++r) {  // run 0 warms up
        float ms = 0.f;
        if (cudaEventRecord(e0, 0) != cudaSuccess) { status = CREDIT_ERR_CUDA; break; }
        stage_copy_kernel<<<(unsigned)ctas, 256, (size_t)fp>>>(s, dd, fpi, err);
        if (cudaGetLastError() != cudaSuccess || cudaEventRecord(e1, 0) != cudaSuccess ||
            cudaEventSynchronize(e1) != cudaSuccess || cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess) {
            cudaGetLastError();
            status = CREDIT_ERR_CUDA;
            break;
        }
        if (r > 0) t.push_back(1e3 * ms);
    }
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    cudaFree(src);
    cudaFree(dst);
    if (status != CREDIT_OK) return status;
    if (credit_get_device_error(device) != CREDIT_OK) return CREDIT_ERR_DEVICE_TIMEOUT;
    *gbps = 2.0 * (double)bytes / median(t) / 1e3;  // bytes / us / 1e3 = GB/s
    return CREDIT_OK;
}
