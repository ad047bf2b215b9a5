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
//       -- or, with the st.async exchange, each push is an st.async whose
//       bytes complete on the receiving CTA's mbarrier, and every CTA waits
//       for its own P - 1 deposits alone; the cluster barrier moves to the
//       kernel's end, where it only keeps CTAs alive until every deposit
//       has landed;
//   a6  fold the P local slots in rank order: every CTA rebuilds the same
//       statistics with local reads only ("All-Gather Trade-off");
//   a7  apply h to the staged slice and write the output slice
//       ("Output Generation").
// A relaxed cluster arrive at kernel entry, waited on just before the push,
// guarantees every peer is running before its shared memory is written.
// With the barrier exchange no CTA touches a peer's shared memory after a5,
// so CTAs may exit without the second barrier (the page's second barrier
// protects slot reuse, which a one-row-per-cluster launch never does).
#include "credit.h"
#include "common.cuh"
#include "internal.h"
#include "rowops.cuh"

namespace credit {

// Phase trace of the checked build: thread 0 of each CTA below kTraceCtas
// stamps %globaltimer at seven points of its life, and its SM id.
constexpr int kTraceCtas = CREDIT_TRACE_CTAS;
#ifdef CREDIT_DEBUG
__device__ unsigned long long g_trace[kTraceCtas][8];
#define CREDIT_TRACE(i)                                                        \
    do {                                                                       \
        if (threadIdx.x == 0 && blockIdx.x < (unsigned)kTraceCtas)             \
            g_trace[blockIdx.x][(i)] = (i) == 7 ? smid() : globaltimer_ns();   \
    } while (0)
#else
#define CREDIT_TRACE(i) \
    do {                \
    } while (0)
#endif

// DEEP: the instantiation for slices that leave room for at most two CTAs
// per SM -- it may use twice the registers, which its pipelined output pass
// spends on twice as many parameter loads in flight per lane.
template <int OP, typename T, typename PT, bool BULK, int R, bool DEEP = false,
          bool QUAD = false>
__global__ void __launch_bounds__(kClusterMaxThreads, DEEP ? 2 : (QUAD ? 4 : 3))
cluster_reduce_reuse(const ClusterArgs a) {
    constexpr int kPipeU = DEEP ? 4 : 2;  // granules per lane in a pipelined output tile
    static_assert(BULK || R == 1, "the element path stages one row per cluster");
    using E = Elem<T>;
    constexpr int VEC = E::kVec;
    extern __shared__ __align__(128) unsigned char stage[];
    __shared__ __align__(16) float slots[kMaxCluster * R * kSlotStride];
    __shared__ __align__(16) float red[2][kMaxWarps * 2 * R];
    __shared__ __align__(8) uint64_t mbar[kMaxChunks];
    __shared__ __align__(8) uint64_t recv_bar;  // st.async exchange: deposits land here

    const uint32_t P = cluster_nctarank();
    const uint32_t rank = cluster_ctarank();
    const bool async_x = a.exchange == 1 && P > 1;
    const int64_t row0 = (blockIdx.x / P) * (int64_t)R;
    const int rows = (int)min((int64_t)R, a.rows - row0);  // live rows of this cluster
    // L2 tail: a CTA may stage only the first a.staged elements of each of
    // its rows' slices; the rest is read from HBM once for the statistics
    // (kept in L2) and once more, from L2, for the output
    constexpr bool kTail = BULK && tail_capable(OP, (int)sizeof(T));
    const int64_t start = (int64_t)rank * a.slice;
    const int n_full = (int)max((int64_t)0, min(a.cols - start, a.slice));
    const int n_slice = kTail ? (int)min((int64_t)n_full, a.staged) : n_full;
    // checked build: the live rows' staged slices and their chunk mbarriers
    // must fit the launch
    const bool fits =
        layout_fits(BULK ? (uint64_t)(rows - 1) * a.pitch + (uint64_t)n_slice * sizeof(T)
                         : (uint64_t)n_slice * sizeof(T),
                    BULK ? (int64_t)rows * ((n_slice + a.chunk_elems - 1) / a.chunk_elems) : 0,
                    kMaxChunks, a.err);
    const int n = fits ? n_slice : 0;                       // staged elements
    const int ntail = kTail && fits ? n_full - n_slice : 0;  // L2-tail elements
    const T* xs = static_cast<const T*>(a.x) + row0 * a.cols + start;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31, nwarps = nt >> 5;
    const int nvec = n / VEC;  // whole 16-byte vectors (all of n on the bulk path)
    CREDIT_TRACE(0);
    CREDIT_TRACE(7);

    if (async_x && threadIdx.x == 0) {
        // the exchange's mbarrier: two arrivals (this one, which registers the
        // P - 1 peers' R deposits of 16 bytes each before any peer can pass
        // the entry barrier below, and the thread that stores this CTA's own
        // partials locally) plus those bytes
        const uint32_t rb = smem_u32(&recv_bar);
        mbar_init(rb, 2);
        mbar_arrive_expect_tx(rb, (P - 1) * R * 16u);
        fence_mbar_init();
    }
    if (P > 1) cluster_arrive_relaxed();

    // ---------------------------------------------------------- a2 stage
    // row i's slice goes to stage + i * pitch, in chunks of chunk_elems with
    // one mbarrier each (row-major chunk numbering)
    int cpr = 1;     // chunks per row
    int vpc = nvec;  // vectors per chunk
    if constexpr (BULK) {
        cpr = (n + a.chunk_elems - 1) / a.chunk_elems;
        vpc = a.chunk_elems / VEC;
        if (tid == 0) {
            const uint32_t st_s = smem_u32(stage);
            for (int c = 0; c < rows * cpr; ++c) mbar_init(smem_u32(&mbar[c]), 1);
            fence_mbar_init();
            fence_proxy_async_smem();
            const uint64_t pol = l2_policy_evict_first();
            for (int i = 0; i < rows; ++i) {
                for (int c = 0; c < cpr; ++c) {
                    const int e0 = c * a.chunk_elems;
                    const uint32_t bytes = (uint32_t)(min(a.chunk_elems, n - e0) * (int)sizeof(T));
                    const uint32_t bar = smem_u32(&mbar[i * cpr + c]);
                    mbar_arrive_expect_tx(bar, bytes);
                    bulk_g2s(st_s + (uint32_t)(i * a.pitch + e0 * (int)sizeof(T)),
                             xs + (int64_t)i * a.cols + e0, bytes, bar, pol);
                }
            }
        }
        __syncthreads();
        CREDIT_TRACE(1);
    } else {
        T* st = reinterpret_cast<T*>(stage);
        for (int i = tid; i < n; i += nt) st[i] = xs[i];
        __syncthreads();
    }
    auto tail_at = [&](int i) { return E::to_f(reinterpret_cast<const T*>(stage)[i]); };

    // --------------------------------------------- a3 local partials
    // each chunk is folded into the threads' statistics as soon as it lands
    // (the L2 tail first, while the bulk copies are in flight)
    const PT* wp = OP == kWStd ? static_cast<const PT*>(a.p0) + start : nullptr;  // weights
    Stats<OP, T> st[R];
    if constexpr (kTail) {
        if (ntail > 0) {
            const uint64_t keep = l2_policy_evict_last();
#pragma unroll
            for (int i = 0; i < R; ++i)
                if (i < rows)
                    stats_global(st[i], reinterpret_cast<const unsigned char*>(xs + i * a.cols + n),
                                 ntail / VEC, warp, nwarps, lane, keep);
        }
    }
#pragma unroll
    for (int i = 0; i < R; ++i) {
        if (i < rows) {
            for (int c = 0; c < cpr; ++c) {
                if constexpr (BULK) mbar_wait_bounded(smem_u32(&mbar[i * cpr + c]), 0, a.err);
                const int v0 = c * vpc;
                if constexpr (OP == kWStd && !BULK) continue;  // weights may be misaligned
                stats_tiles(st[i], stage + (size_t)i * a.pitch + (size_t)v0 * 16,
                            min(nvec, v0 + vpc) - v0, warp, nwarps, lane,
                            wp ? wp + (int64_t)v0 * VEC : wp);
            }
        }
    }
    if constexpr (!BULK) {
        if constexpr (OP == kWStd) {
            for (int i = tid; i < n; i += nt) st[0].add1(tail_at(i), load_param1<PT>(wp, i));
        } else {
            for (int i = nvec * VEC + tid; i < n; i += nt) st[0].add1(tail_at(i));
        }
    }
    CREDIT_TRACE(2);
    auto stash = [&](int i, float mq) {
        float s = softmax_stash(stage + (size_t)i * a.pitch, nvec, warp, nwarps, lane, mq);
        if constexpr (!BULK) {
            for (int e = nvec * VEC + tid; e < n; e += nt) {
                const float t = expf(tail_at(e) - mq);
                reinterpret_cast<float*>(stage)[e] = t;
                s += t;
            }
        }
        return s;
    };
    float p[R][3];
    cta_partial_rows<OP, T, R>(st, red[0], red[1], nwarps, nt, stash, p);
    CREDIT_TRACE(3);

    // --------------------------------------- a4 push, a5 barrier, a6 combine
    float stv[R][3];  // combined statistics, identical in every CTA of the cluster
#pragma unroll
    for (int i = 0; i < R; ++i) { stv[i][0] = p[i][0]; stv[i][1] = p[i][1]; stv[i][2] = p[i][2]; }
    if (P > 1) {
        cluster_wait_acquire();  // every peer has started: its slots (and mbarrier) exist
        if (async_x) {
            // thread t deposits into peer t (each deposit counts 16 bytes on
            // that peer's mbarrier); thread `rank` stores locally and arrives
            if (tid == (int)rank) {
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    float* d = &slots[(rank * R + i) * kSlotStride];
                    d[0] = p[i][0]; d[1] = p[i][1]; d[2] = p[i][2];
                }
                mbar_arrive(smem_u32(&recv_bar));
            } else if (tid < (int)P) {
                const uint32_t rbar = mapa_shared(smem_u32(&recv_bar), (uint32_t)tid);
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    const uint32_t dst =
                        mapa_shared(smem_u32(&slots[(rank * R + i) * kSlotStride]), (uint32_t)tid);
                    st_async_v4f32(dst, p[i][0], p[i][1], p[i][2], 0.f, rbar);
                }
            }
            mbar_wait_bounded(smem_u32(&recv_bar), 0, a.err);  // all P partials are here
            cluster_arrive_relaxed();  // nothing more lands in this CTA's shared memory
        } else {
            if (tid < (int)P) {
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    const uint32_t dst =
                        mapa_shared(smem_u32(&slots[(rank * R + i) * kSlotStride]), (uint32_t)tid);
                    st_cluster_v4f32(dst, p[i][0], p[i][1], p[i][2], 0.f);
                }
            }
            cluster_arrive_release();
            cluster_wait_acquire();
        }
#pragma unroll
        for (int i = 0; i < R; ++i) {
            combine_slots_strided<OP>(slots + i * kSlotStride, P, R * kSlotStride, stv[i][0],
                                      stv[i][1], stv[i][2]);
        }
    }

    if (tid == 0) {
        for (int i = 0; i < rows; ++i) debug_row_stats(a.dbg_stats, row0 + i, rank, P, stv[i], 3);
    }
    CREDIT_TRACE(4);
    // ------------------------------------------------------- a7 output
    constexpr bool kParams = OP == kLayerNorm || OP == kRMSNorm;
    const PT* g = kParams ? static_cast<const PT*>(a.p0) : nullptr;
    const PT* b = kParams ? static_cast<const PT*>(a.p1) : nullptr;
    OutputMap<OP, T> h[R];
#pragma unroll
    for (int i = 0; i < R; ++i) h[i] = OutputMap<OP, T>(stv[i][0], stv[i][1], stv[i][2], p[i][0], a.cols, a.eps);
    if constexpr (OP == kQuant) {
        int8_t* qrow[R];
#pragma unroll
        for (int i = 0; i < R; ++i) qrow[i] = static_cast<int8_t*>(a.y) + (row0 + i) * a.cols + start;
        if (rank == 0 && tid == 0)
            for (int i = 0; i < rows; ++i) a.aux[row0 + i] = h[i].c0;  // the row scales
        if constexpr (BULK) {
            output_quant_rows<T, R>(h, stage, a.pitch, qrow, rows, nvec, warp, nwarps, lane);
        } else {
            for (int i = tid; i < n; i += nt) qrow[0][i] = (int8_t)h[0].code(tail_at(i));
        }
    } else {
        T* yrow[R];
#pragma unroll
        for (int i = 0; i < R; ++i) yrow[i] = static_cast<T*>(a.y) + (row0 + i) * a.cols + start;
        // RMSNorm with bf16 data and bf16 weights gains from the pipelined
        // pass (measured); the other operator / type combinations do not
        constexpr bool kPipe = BULK && R == 1 && OP == kRMSNorm && Granule<OP, T, PT>::kPairs == 4;
        // the tail of a slice with 16-byte granules is written from each
        // warp's ring of freed staged tiles; RMSNorm's pipelined pass, which
        // keeps its weight loads ahead of its tiles, and 8-byte granules
        // (bf16 data with fp32 parameters, copied 8 bytes at a time) measured
        // faster with the tail loaded through registers
        constexpr bool kRing = kTail && R == 1 && Granule<OP, T, PT>::kBytes == 16 && !kPipe;
        bool done = false;
        if constexpr (kRing) {
            if (ntail > 0) {
                // staged tiles first, then the tail from each warp's ring
                // (8 KB of each warp in flight)
                constexpr int kRingD = (OP != kSoftmax && Granule<OP, T, PT>::kPairs == 4) ? 8 : 4;
                output_ring<OP, T, PT, kRingD>(
                    h[0], stage, reinterpret_cast<const unsigned char*>(xs + n), yrow[0],
                    g ? g + start : nullptr, b ? b + start : nullptr, nvec, ntail / VEC, warp,
                    nwarps, lane, l2_policy_evict_first());
                done = true;
            }
        }
        if (done) {
        } else if constexpr (kTail) {
            // the L2 tail first: its lines leave L2 as early as possible
            if (ntail > 0) {
                if constexpr (R == 1) {
                    output_tiles<OP, T, PT, NoRelease, false, true>(
                        h[0], reinterpret_cast<const unsigned char*>(xs + n), yrow[0] + n,
                        g ? g + start + n : nullptr, b ? b + start + n : nullptr, ntail / VEC,
                        warp, nwarps, lane, NoRelease(), l2_policy_evict_first());
                } else {
                    T* ytail[R];
#pragma unroll
                    for (int i = 0; i < R; ++i) ytail[i] = yrow[i] + n;
                    output_tiles_rows<OP, T, PT, R, true>(
                        h, reinterpret_cast<const unsigned char*>(xs + n),
                        a.cols * (int64_t)sizeof(T), ytail, rows, g ? g + start + n : nullptr,
                        b ? b + start + n : nullptr, ntail / VEC, warp, nwarps, lane,
                        l2_policy_evict_first());
                }
            }
        }
        if (done) {
        } else if constexpr (kPipe) {
            if (g) {
                output_tiles_pipelined<OP, T, PT, kPipeU>(h[0], stage, yrow[0], g + start, nullptr,
                                                          nvec, warp, nwarps, lane);
            } else {
                output_tiles_rows<OP, T, PT, R>(h, stage, a.pitch, yrow, rows, nullptr, nullptr,
                                                nvec, warp, nwarps, lane);
            }
        } else if constexpr (BULK) {
            output_tiles_rows<OP, T, PT, R>(h, stage, a.pitch, yrow, rows, g ? g + start : nullptr,
                                            b ? b + start : nullptr, nvec, warp, nwarps, lane);
        } else {
            for (int i = tid; i < n; i += nt) {
                const float gj = g ? load_param1<PT>(g, start + i) : 1.f;
                const float bj = b ? load_param1<PT>(b, start + i) : 0.f;
                yrow[0][i] = E::from_f(h[0].one(tail_at(i), gj, bj));
            }
        }
    }
    CREDIT_TRACE(5);
    // st.async exchange: a peer arrives only once all deposits to it have
    // landed, so when this completes every deposit in the cluster has, and
    // no CTA leaves while one is in flight
    if (async_x) cluster_wait_acquire();
    CREDIT_TRACE(6);
}

// ----------------------------------------------------------- dispatch
template <int OP, typename T, typename PT>
static const void* pick_rows(bool vec, int rows, bool deep = false, bool quad = false) {
    if (!vec) return rows == 1 ? (const void*)cluster_reduce_reuse<OP, T, PT, false, 1> : nullptr;
    // the deep instantiation exists where the output pass is pipelined
    constexpr bool kHasDeep = OP == kRMSNorm && Granule<OP, T, PT>::kPairs == 4;
    if constexpr (kHasDeep) {
        if (deep && rows == 1) return (const void*)cluster_reduce_reuse<OP, T, PT, true, 1, true>;
    }
    // the four-CTA instantiation (64 registers)
    if constexpr (quad_capable(OP, (int)sizeof(T), (int)sizeof(PT))) {
        if (quad && rows == 1)
            return (const void*)cluster_reduce_reuse<OP, T, PT, true, 1, false, true>;
    }
    switch (rows) {
        case 1: return (const void*)cluster_reduce_reuse<OP, T, PT, true, 1>;
        case 2: return (const void*)cluster_reduce_reuse<OP, T, PT, true, 2>;
        case 4: return (const void*)cluster_reduce_reuse<OP, T, PT, true, 4>;
    }
    return nullptr;
}

template <int OP, typename T>
static const void* pick_param(int pdtype, bool vec, int rows, bool deep, bool quad) {
    return pdtype == 0 ? pick_rows<OP, T, float>(vec, rows, deep, quad)
                       : pick_rows<OP, T, bf16>(vec, rows, deep, quad);
}

template <int OP>
static const void* pick_dtype(int dtype, int pdtype, bool vec, int rows, bool deep = false,
                              bool quad = false) {
    return dtype == 0 ? pick_param<OP, float>(pdtype, vec, rows, deep, quad)
                      : pick_param<OP, bf16>(pdtype, vec, rows, deep, quad);
}

const void* cluster_kernel(KernelKey k) {
    switch (k.op) {
        case kSoftmax: return k.dtype == 0 ? pick_rows<kSoftmax, float, float>(k.vec, k.rows)
                                           : pick_rows<kSoftmax, bf16, float>(k.vec, k.rows,
                                                                              false, k.quad);
        case kLayerNorm:
            return pick_dtype<kLayerNorm>(k.dtype, k.pdtype, k.vec, k.rows, false, k.quad);
        case kRMSNorm:
            return pick_dtype<kRMSNorm>(k.dtype, k.pdtype, k.vec, k.rows, k.deep, k.quad);
        case kQuant: return k.dtype == 0 ? pick_rows<kQuant, float, float>(k.vec, k.rows)
                                         : pick_rows<kQuant, bf16, float>(k.vec, k.rows);
        case kWStd: return pick_dtype<kWStd>(k.dtype, k.pdtype, k.vec, k.rows);
        case kPearson: return k.rows == 1 ? pearson_cluster_kernel(k.dtype, k.vec) : nullptr;
    }
    return nullptr;
}

cudaError_t launch_cluster(KernelKey k, const ClusterArgs& a, int P, int threads, size_t smem,
                           cudaStream_t s) {
    const void* fn = cluster_kernel(k);
    if (!fn) return cudaErrorInvalidDeviceFunction;
    const size_t esz = k.dtype == 0 ? 4 : 2;
    const size_t yesz = k.op == kQuant ? 1 : esz;  // int8 codes
    // gridDim.x is limited to 2^31 - 1: launch in batches of whole clusters
    const int64_t max_rows = (int64_t)(0x7fffffff / P) * k.rows;
    for (int64_t r0 = 0; r0 < a.rows; r0 += max_rows) {
        const int64_t nr = a.rows - r0 < max_rows ? a.rows - r0 : max_rows;
        ClusterArgs b = a;
        b.x = static_cast<const char*>(a.x) + r0 * a.cols * (int64_t)esz;
        b.y = static_cast<char*>(a.y) + r0 * a.cols * (int64_t)yesz;
        if (a.aux) b.aux = a.aux + r0;
        if (k.op == kPearson) b.p0 = static_cast<const char*>(a.p0) + r0 * a.cols * (int64_t)esz;
        b.rows = nr;
        const int64_t nclusters = (nr + k.rows - 1) / k.rows;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(nclusters * P), 1, 1);
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

extern "C" credit_status_t credit_debug_trace(void* host, int64_t ctas) {
#ifdef CREDIT_DEBUG
    if (!host || ctas < 1 || ctas > credit::kTraceCtas) return CREDIT_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpyFromSymbol(host, credit::g_trace, (size_t)ctas * 64) != cudaSuccess) {
        cudaGetLastError();
        return CREDIT_ERR_CUDA;
    }
    return CREDIT_OK;
#else
    (void)host;
    (void)ctas;
    return CREDIT_ERR_UNSUPPORTED;
#endif
}
