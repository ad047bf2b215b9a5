// cluster.cu -- the clustered DSMEM reduce-reuse kernel.
//
// Protocol (CREDIT summary page, arXiv 2609.01864v1, "C. Cluster Reduction
// and Reuse Protocol"), one row per cluster of P CTAs, CTA `rank` owning the
// contiguous slice [rank * slice, (rank + 1) * slice) of the row:
//   a2  stage the slice into shared memory once (bulk copies, one mbarrier
//       per chunk, or element loads on the unaligned path);
//   a3  reduce it to a compact partial: thread accumulation, warp shuffles,
//       a shared-memory fold ("Partial Reduction");
//   a4  push the partial into slot `rank` of every peer's slot array with
//       mapa + st.shared::cluster ("Replicated Push");
//   a5  cluster barrier (arrive.release / wait.acquire) makes the pushes
//       visible ("Synchronization");
//   a6  fold the P local slots in rank order: every CTA rebuilds the same
//       statistics with local reads only ("All-Gather Trade-off");
//   a7  apply h to the staged slice and write the output slice
//       ("Output Generation").
// A relaxed cluster arrive at kernel entry, waited on just before the push,
// guarantees every peer is running before its shared memory is written.
// After barrier a5 no CTA touches a peer's shared memory, so CTAs may exit
// without the second barrier (the page's second barrier protects slot reuse,
// which a one-row-per-cluster launch never does).
#include "common.cuh"
#include "internal.h"
#include "rowops.cuh"

namespace credit {

template <int OP, typename T, typename PT, bool BULK>
__global__ void __launch_bounds__(kMaxThreads, 2)
cluster_reduce_reuse(const ClusterArgs a) {
    using E = Elem<T>;
    constexpr int VEC = E::kVec;
    extern __shared__ __align__(128) unsigned char stage[];
    __shared__ __align__(16) float slots[kMaxCluster * kSlotStride];
    __shared__ __align__(16) float red[2][kMaxWarps * 2];
    __shared__ __align__(8) uint64_t mbar[kMaxChunks];

    const uint32_t P = cluster_nctarank();
    const uint32_t rank = cluster_ctarank();
    const int64_t row = blockIdx.x / P;
    const int64_t start = (int64_t)rank * a.slice;
    const int n = (int)max((int64_t)0, min(a.cols - start, a.slice));
    const T* xs = static_cast<const T*>(a.x) + row * a.cols + start;
    T* ys = static_cast<T*>(a.y) + row * a.cols + start;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int nvec = n / VEC;  // whole 16-byte vectors (all of n on the bulk path)

    if (P > 1) cluster_arrive_relaxed();

    // ---------------------------------------------------------- a2 stage
    int nchunks = 1;
    int vpc = nvec;  // vectors per chunk
    if constexpr (BULK) {
        nchunks = (n + a.chunk_elems - 1) / a.chunk_elems;
        vpc = a.chunk_elems / VEC;
        if (tid == 0) {
            const uint32_t st_s = smem_u32(stage);
            for (int c = 0; c < nchunks; ++c) mbar_init(smem_u32(&mbar[c]), 1);
            fence_mbar_init();
            fence_proxy_async_smem();
            const uint64_t pol = l2_policy_evict_first();
            for (int c = 0; c < nchunks; ++c) {
                const int e0 = c * a.chunk_elems;
                const uint32_t bytes = (uint32_t)(min(a.chunk_elems, n - e0) * (int)sizeof(T));
                const uint32_t bar = smem_u32(&mbar[c]);
                mbar_arrive_expect_tx(bar, bytes);
                bulk_g2s(st_s + (uint32_t)(e0 * (int)sizeof(T)), xs + e0, bytes, bar, pol);
            }
        }
        __syncthreads();
    } else {
        T* st = reinterpret_cast<T*>(stage);
        for (int i = tid; i < n; i += nt) st[i] = xs[i];
        __syncthreads();
    }
    auto tail_at = [&](int i) { return E::to_f(reinterpret_cast<const T*>(stage)[i]); };

    // --------------------------------------------- a3 local partial
    // each chunk is folded into the threads' statistics as soon as it lands
    const int warp = tid >> 5, lane = tid & 31, nwarps = nt >> 5;
    Stats<OP, T> st;
    for (int c = 0; c < nchunks; ++c) {
        if constexpr (BULK) mbar_wait_bounded(smem_u32(&mbar[c]), 0, a.err);
        const int v0 = c * vpc;
        stats_tiles(st, stage + (size_t)v0 * 16, min(nvec, v0 + vpc) - v0, warp, nwarps, lane);
    }
    if constexpr (!BULK)
        for (int i = nvec * VEC + tid; i < n; i += nt) st.add1(tail_at(i));
    auto stash = [&](float mq) {
        float s = softmax_stash(stage, nvec, warp, nwarps, lane, mq);
        if constexpr (!BULK) {
            for (int i = nvec * VEC + tid; i < n; i += nt) {
                const float t = expf(tail_at(i) - mq);
                reinterpret_cast<float*>(stage)[i] = t;
                s += t;
            }
        }
        return s;
    };
    float p0, p1, p2;
    cta_partial<OP, T>(st, red[0], red[1], nwarps, nt, stash, p0, p1, p2);

    // --------------------------------------- a4 push, a5 barrier, a6 combine
    float st0 = p0, st1 = p1, st2 = p2;  // combined statistics, identical in every CTA
    if (P > 1) {
        cluster_wait_acquire();  // every peer has started: its slots exist
        if (tid < (int)P) {
            const uint32_t dst = mapa_shared(smem_u32(&slots[rank * kSlotStride]), (uint32_t)tid);
            st_cluster_v4f32(dst, p0, p1, p2, 0.f);
        }
        cluster_arrive_release();
        cluster_wait_acquire();
        combine_slots<OP>(slots, P, st0, st1, st2);
    }

    // ------------------------------------------------------- a7 output
    const OutputMap<OP, T> h(st0, st1, st2, p0, a.cols, a.eps);
    const PT* g = static_cast<const PT*>(a.p0);
    const PT* b = static_cast<const PT*>(a.p1);
    if constexpr (BULK) {
        output_tiles<OP, T, PT>(h, stage, ys, g ? g + start : nullptr, b ? b + start : nullptr,
                                nvec, warp, nwarps, lane);
    } else {
        for (int i = tid; i < n; i += nt) {
            const float gj = (OP != kSoftmax && g) ? load_param1<PT>(g, start + i) : 1.f;
            const float bj = (OP != kSoftmax && b) ? load_param1<PT>(b, start + i) : 0.f;
            ys[i] = E::from_f(h.one(tail_at(i), gj, bj));
        }
    }
}

// ----------------------------------------------------------- dispatch
template <int OP, typename T, typename PT>
static const void* pick_bulk(bool vec) {
    return vec ? (const void*)cluster_reduce_reuse<OP, T, PT, true>
               : (const void*)cluster_reduce_reuse<OP, T, PT, false>;
}

template <int OP, typename T>
static const void* pick_param(int pdtype, bool vec) {
    return pdtype == 0 ? pick_bulk<OP, T, float>(vec) : pick_bulk<OP, T, bf16>(vec);
}

template <int OP>
static const void* pick_dtype(int dtype, int pdtype, bool vec) {
    return dtype == 0 ? pick_param<OP, float>(pdtype, vec) : pick_param<OP, bf16>(pdtype, vec);
}

const void* cluster_kernel(KernelKey k) {
    switch (k.op) {
        case kSoftmax: return k.dtype == 0 ? pick_bulk<kSoftmax, float, float>(k.vec)
                                           : pick_bulk<kSoftmax, bf16, float>(k.vec);
        case kLayerNorm: return pick_dtype<kLayerNorm>(k.dtype, k.pdtype, k.vec);
        case kRMSNorm: return pick_dtype<kRMSNorm>(k.dtype, k.pdtype, k.vec);
    }
    return nullptr;
}

cudaError_t launch_cluster(KernelKey k, const ClusterArgs& a, int64_t rows, int P,
                           int threads, size_t smem, cudaStream_t s) {
    const void* fn = cluster_kernel(k);
    if (!fn) return cudaErrorInvalidDeviceFunction;
    const size_t esz = k.dtype == 0 ? 4 : 2;
    // gridDim.x is limited to 2^31 - 1: launch in row batches.
    const int64_t max_rows = (int64_t)(0x7fffffff / P);
    for (int64_t r0 = 0; r0 < rows; r0 += max_rows) {
        const int64_t nr = rows - r0 < max_rows ? rows - r0 : max_rows;
        ClusterArgs b = a;
        b.x = static_cast<const char*>(a.x) + r0 * a.cols * (int64_t)esz;
        b.y = static_cast<char*>(a.y) + r0 * a.cols * (int64_t)esz;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(nr * P), 1, 1);
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
        void* args[] = {&b};
        cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace credit
