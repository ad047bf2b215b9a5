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

namespace credit {

template <int OP, typename T, typename PT, bool BULK>
__global__ void __launch_bounds__(kMaxThreads, 1)
cluster_reduce_reuse(const ClusterArgs a) {
    using E = Elem<T>;
    constexpr int VEC = E::kVec;
    extern __shared__ __align__(128) unsigned char stage[];
    __shared__ __align__(16) float slots[kMaxCluster * kSlotStride];
    __shared__ float red[2][kMaxWarps];
    __shared__ __align__(8) uint64_t mbar[kMaxChunks];

    const uint32_t P = cluster_nctarank();
    const uint32_t rank = cluster_ctarank();
    const int64_t row = blockIdx.x / P;
    const int64_t start = (int64_t)rank * a.slice;
    const int64_t n = max((int64_t)0, min(a.cols - start, a.slice));
    const T* xs = static_cast<const T*>(a.x) + row * a.cols + start;
    T* ys = static_cast<T*>(a.y) + row * a.cols + start;
    const int tid = threadIdx.x, nt = blockDim.x;
    const uint32_t st_s = smem_u32(stage);
    const int64_t nvec = n / VEC;  // whole 16-byte vectors (all of n on the bulk path)

    if (P > 1) cluster_arrive_relaxed();

    // ---------------------------------------------------------- a2 stage
    int nchunks = 1;
    int64_t vpc = nvec;  // vectors per chunk
    if constexpr (BULK) {
        nchunks = (int)((n + a.chunk_elems - 1) / a.chunk_elems);
        vpc = a.chunk_elems / VEC;
        if (tid == 0) {
            for (int c = 0; c < nchunks; ++c) mbar_init(smem_u32(&mbar[c]), 1);
            fence_mbar_init();
            fence_proxy_async_smem();
            const uint64_t pol = l2_policy_evict_first();
            for (int c = 0; c < nchunks; ++c) {
                const int64_t e0 = (int64_t)c * a.chunk_elems;
                const uint32_t bytes =
                    (uint32_t)(min((int64_t)a.chunk_elems, n - e0) * (int64_t)sizeof(T));
                const uint32_t bar = smem_u32(&mbar[c]);
                mbar_arrive_expect_tx(bar, bytes);
                bulk_g2s(st_s + (uint32_t)(e0 * sizeof(T)), xs + e0, bytes, bar, pol);
            }
        }
        __syncthreads();
    } else {
        T* st = reinterpret_cast<T*>(stage);
        for (int64_t i = tid; i < n; i += nt) st[i] = xs[i];
        __syncthreads();
    }

    auto vec_at = [&](int64_t v, float* f) { E::unpack(ld_shared_v4(st_s + (uint32_t)(v * 16)), f); };
    auto tail_at = [&](int64_t i) { return E::to_f(reinterpret_cast<const T*>(stage)[i]); };

    // -------------------------------------------- a3 local partial, pass A
    // max (softmax), sum (LayerNorm) or sum of squares (RMSNorm), consumed
    // chunk by chunk as the bulk copies land.
    float acc = (OP == kSoftmax) ? -INFINITY : 0.f;
    for (int c = 0; c < nchunks; ++c) {
        if constexpr (BULK) mbar_wait_bounded(smem_u32(&mbar[c]), 0, a.err);
        const int64_t vend = min(nvec, (int64_t)(c + 1) * vpc);
        for (int64_t v = (int64_t)c * vpc + tid; v < vend; v += nt) {
            float f[VEC];
            vec_at(v, f);
#pragma unroll
            for (int k = 0; k < VEC; ++k) {
                if constexpr (OP == kSoftmax) acc = fmaxf(acc, f[k]);
                else if constexpr (OP == kLayerNorm) acc += f[k];
                else acc = fmaf(f[k], f[k], acc);
            }
        }
    }
    if constexpr (!BULK) {
        for (int64_t i = nvec * VEC + tid; i < n; i += nt) {
            const float f = tail_at(i);
            if constexpr (OP == kSoftmax) acc = fmaxf(acc, f);
            else if constexpr (OP == kLayerNorm) acc += f;
            else acc = fmaf(f, f, acc);
        }
    }
    float pv0, pv1 = 0.f, pv2 = 0.f;
    if constexpr (OP == kSoftmax) pv0 = block_allreduce(acc, red[0], MaxOp{}, -INFINITY);
    else pv0 = block_allreduce(acc, red[0], SumOp{}, 0.f);

    // -------------------------------------------------------- pass B
    if constexpr (OP == kSoftmax) {
        // s_q = sum exp(x - m_q); fp32 keeps t = exp(x - m_q) in place so the
        // output pass is a single multiply.
        const float mq = pv0, mq_l2e = mq * kLog2e;
        float s = 0.f;
        if (n > 0) {
            for (int64_t v = tid; v < nvec; v += nt) {
                float f[VEC];
                vec_at(v, f);
#pragma unroll
                for (int k = 0; k < VEC; ++k) {
                    f[k] = exp_shift<T>(f[k], mq, mq_l2e);
                    s += f[k];
                }
                if constexpr (sizeof(T) == 4) st_shared_v4(st_s + (uint32_t)(v * 16), E::pack(f));
            }
            if constexpr (!BULK) {
                for (int64_t i = nvec * VEC + tid; i < n; i += nt) {
                    const float t = exp_shift<T>(tail_at(i), mq, mq_l2e);
                    s += t;
                    if constexpr (sizeof(T) == 4) reinterpret_cast<float*>(stage)[i] = t;
                }
            }
        }
        pv1 = block_allreduce(s, red[1], SumOp{}, 0.f);
    } else if constexpr (OP == kLayerNorm) {
        // exact two-pass over the staged slice: (n_q, mean_q, M2_q)
        const float nq = (float)n;
        const float mu = n > 0 ? pv0 / nq : 0.f;
        float m2 = 0.f;
        for (int64_t v = tid; v < nvec; v += nt) {
            float f[VEC];
            vec_at(v, f);
#pragma unroll
            for (int k = 0; k < VEC; ++k) {
                const float d = f[k] - mu;
                m2 = fmaf(d, d, m2);
            }
        }
        if constexpr (!BULK) {
            for (int64_t i = nvec * VEC + tid; i < n; i += nt) {
                const float d = tail_at(i) - mu;
                m2 = fmaf(d, d, m2);
            }
        }
        pv1 = mu;
        pv2 = block_allreduce(m2, red[1], SumOp{}, 0.f);
        pv0 = nq;
    }

    // --------------------------------------- a4 push, a5 barrier, a6 combine
    float st0, st1, st2;  // combined statistics, identical in every CTA
    if (P > 1) {
        cluster_wait_acquire();  // every peer has started: its slots exist
        if (tid < (int)P) {
            const uint32_t dst = mapa_shared(smem_u32(&slots[rank * kSlotStride]), (uint32_t)tid);
            st_cluster_v4f32(dst, pv0, pv1, pv2, 0.f);
        }
        cluster_arrive_release();
        cluster_wait_acquire();
        if constexpr (OP == kSoftmax) {
            float m = -INFINITY;
            for (uint32_t q = 0; q < P; ++q) m = fmaxf(m, slots[q * kSlotStride]);
            float s = 0.f;
            for (uint32_t q = 0; q < P; ++q)
                s += rescale(slots[q * kSlotStride + 1], slots[q * kSlotStride], m);
            st0 = m; st1 = s; st2 = 0.f;
        } else if constexpr (OP == kLayerNorm) {
            NormPart acc2{0.f, 0.f, 0.f};
            for (uint32_t q = 0; q < P; ++q)
                acc2 = chan_merge(acc2, NormPart{slots[q * kSlotStride], slots[q * kSlotStride + 1],
                                                 slots[q * kSlotStride + 2]});
            st0 = acc2.n; st1 = acc2.mu; st2 = acc2.m2;
        } else {
            float ss = 0.f;
            for (uint32_t q = 0; q < P; ++q) ss += slots[q * kSlotStride];
            st0 = ss; st1 = st2 = 0.f;
        }
    } else {
        st0 = pv0; st1 = pv1; st2 = pv2;
    }

    // ------------------------------------------------------- a7 output
    const float inv_n = 1.f / (float)a.cols;
    float c0 = 0.f, c1 = 0.f;
    if constexpr (OP == kSoftmax) {
        if constexpr (sizeof(T) == 4) c0 = rescale(1.f, pv0, st0) / st1;  // exp(m_q - m) / s
        else { c0 = st0 * kLog2e; c1 = 1.f / st1; }
    } else if constexpr (OP == kLayerNorm) {
        c0 = st1;                                        // mean
        c1 = 1.f / sqrtf(fmaxf(st2 * inv_n, 0.f) + a.eps);  // 1 / sqrt(var + eps)
    } else {
        c0 = 1.f / sqrtf(st0 * inv_n + a.eps);
    }
    const PT* g = static_cast<const PT*>(a.p0);
    const PT* b = static_cast<const PT*>(a.p1);

    auto h = [&](float f, float gj, float bj) -> float {
        if constexpr (OP == kSoftmax) {
            if constexpr (sizeof(T) == 4) return f * c0;
            else return fast_ex2(fmaf(f, kLog2e, -c0)) * c1;
        } else if constexpr (OP == kLayerNorm) {
            return fmaf((f - c0) * c1, gj, bj);
        } else {
            return (f * c0) * gj;
        }
    };

    for (int64_t v = tid; v < nvec; v += nt) {
        float f[VEC], gv[VEC], bv[VEC];
        vec_at(v, f);
        const int64_t j0 = start + v * VEC;
#pragma unroll
        for (int k = 0; k < VEC; ++k) { gv[k] = 1.f; bv[k] = 0.f; }
        if constexpr (OP != kSoftmax) {
            if constexpr (BULK) {
                if (g) load_params<PT, VEC>(g, j0, gv);
                if (b) load_params<PT, VEC>(b, j0, bv);
            } else {
#pragma unroll
                for (int k = 0; k < VEC; ++k) {
                    if (g) gv[k] = load_param1<PT>(g, j0 + k);
                    if (b) bv[k] = load_param1<PT>(b, j0 + k);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < VEC; ++k) f[k] = h(f[k], gv[k], bv[k]);
        if constexpr (BULK) {
            st_global_cs_v4(ys + v * VEC, E::pack(f));
        } else {
#pragma unroll
            for (int k = 0; k < VEC; ++k) ys[v * VEC + k] = E::from_f(f[k]);
        }
    }
    if constexpr (!BULK) {
        for (int64_t i = nvec * VEC + tid; i < n; i += nt) {
            const float gj = (OP != kSoftmax && g) ? load_param1<PT>(g, start + i) : 1.f;
            const float bj = (OP != kSoftmax && b) ? load_param1<PT>(b, start + i) : 0.f;
            ys[i] = E::from_f(h(tail_at(i), gj, bj));
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
