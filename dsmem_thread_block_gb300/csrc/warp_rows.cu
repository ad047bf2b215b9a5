// warp_rows.cu -- rows short enough for one warp's registers.
//
// The reduce-then-reuse pattern at warp scope: a warp loads a whole row (each
// lane up to kWarpRowNV coalesced 16-byte vectors), reduces it with warp
// shuffles, applies h to the values still in its registers and writes the
// row -- one HBM read and one write per element, as in the clustered kernel,
// with the reuse held in registers instead of shared memory and no bulk-copy
// setup, mbarrier or block barrier per row.  A grid of resident CTAs strides
// over the rows, one row per warp at a time.  It is the non-clustered
// variant for the narrow end of the CREDIT summary page's width sweep ("D.
// Profitability and Candidate Selection": the baseline for rows a CTA can
// hold), where one CTA per row leaves its per-CTA staging costs exposed.
// Statistics and h are those of the clustered kernel (Stats, OutputMap) with
// P = 1: the warp's partial is the row's.
#include "common.cuh"
#include "internal.h"
#include "rowops.cuh"

namespace credit {

// NV: vectors per lane the instantiation holds (kWarpRowNV, or half of it
// for the norms' rows of at most 2 KiB, whose smaller register footprint
// leaves room for more resident warps: measured faster for LayerNorm and
// RMSNorm, slower for softmax, which keeps the full size).
template <int OP, typename T, typename PT, int NV>
__global__ void __launch_bounds__(kWarpRowThreads)
warp_rows(const WarpRowsArgs a) {
    using E = Elem<T>;
    constexpr int VEC = E::kVec;
    constexpr int NP = VEC / 2;  // element pairs per vector
    constexpr bool kParams = OP == kLayerNorm || OP == kRMSNorm;
    const int lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    const int64_t nw = (int64_t)gridDim.x * wpb;
    const int nvec = (int)(a.cols / VEC);
    const PT* gp = static_cast<const PT*>(a.p0);
    const PT* bp = static_cast<const PT*>(a.p1);

    for (int64_t row = (int64_t)blockIdx.x * wpb + (threadIdx.x >> 5); row < a.rows; row += nw) {
        const T* xr = static_cast<const T*>(a.x) + row * a.cols;
        uint4 v[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int q = lane + 32 * i;
            if (q < nvec) v[i] = ld_global_cs_v4(reinterpret_cast<const uint4*>(xr) + q);
        }
        Stats<OP, T> st;
#pragma unroll
        for (int i = 0; i < NV; ++i)
            if (lane + 32 * i < nvec) st.add(v[i]);

        // the row's statistics, identical in every lane (butterfly shuffles)
        float st0 = 0.f, st1 = 0.f, st2 = 0.f, mq = 0.f;
        if constexpr (OP == kSoftmax && sizeof(T) == 4) {
            // max, then t = exp(x - m) kept in the registers and summed
            const float m = warp_allreduce(st.m, MaxOp());
            F2 s = {0.f, 0.f};
            if (m != -INFINITY) {
#pragma unroll
                for (int i = 0; i < NV; ++i) {
                    if (lane + 32 * i < nvec) {
                        const F2 t0 = {expf(__uint_as_float(v[i].x) - m),
                                       expf(__uint_as_float(v[i].y) - m)};
                        const F2 t1 = {expf(__uint_as_float(v[i].z) - m),
                                       expf(__uint_as_float(v[i].w) - m)};
                        s = add2(s, add2(t0, t1));
                        v[i] = make_uint4(__float_as_uint(t0.x), __float_as_uint(t0.y),
                                          __float_as_uint(t1.x), __float_as_uint(t1.y));
                    }
                }
            }
            st0 = m;
            st1 = warp_allreduce(s.x + s.y, SumOp());
            mq = m;
        } else if constexpr (OP == kSoftmax) {
            const float m = warp_allreduce(st.m, MaxOp());
            st0 = m;
            st1 = warp_allreduce(rescale(st.s.x + st.s.y, st.m, m), SumOp());
            mq = m;
        } else if constexpr (OP == kLayerNorm) {
            // (n, mean, M2) by the parallel-axis form of Chan et al.'s merge
            const float s1 = st.s1.x + st.s1.y, s2 = st.s2.x + st.s2.y;
            const float mt = st.n > 0.f ? s1 / st.n - st.nK.x : 0.f;
            const float m2t = st.n > 0.f ? fmaxf(s2 - s1 * (s1 / st.n), 0.f) : 0.f;
            const float n = warp_allreduce(st.n, SumOp());
            const float mean = n > 0.f ? warp_allreduce(st.n * mt, SumOp()) / n : 0.f;
            const float d = mt - mean;
            st0 = n;
            st1 = mean;
            st2 = warp_allreduce(fmaf(st.n * d, d, m2t), SumOp());
        } else {
            st0 = warp_allreduce(st.q.x + st.q.y, SumOp());
        }
        const OutputMap<OP, T> h(st0, st1, st2, mq, a.cols, a.eps);

        T* yr = static_cast<T*>(a.y) + row * a.cols;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int q = lane + 32 * i;
            if (q < nvec) {
                F2 p[NP];
                Pairs<T>::unpack(v[i], p);
                if constexpr (kParams) {
                    F2 g[NP], b[NP];
                    load_param_pairs<PT, NP>(gp, (int64_t)q * VEC, g, 1.f);
                    load_param_pairs<PT, NP>(bp, (int64_t)q * VEC, b, 0.f);
#pragma unroll
                    for (int j = 0; j < NP; ++j) p[j] = h(p[j], g[j], b[j]);
                } else {
#pragma unroll
                    for (int j = 0; j < NP; ++j) p[j] = h(p[j], p[j], p[j]);
                }
                stg16_stream(reinterpret_cast<uint4*>(yr) + q, Pairs<T>::pack(p));
            }
        }
    }
}

// ----------------------------------------------------------- dispatch
template <int OP, typename T, int NV>
static const void* wr_param(int pdtype) {
    return pdtype == 0 ? (const void*)warp_rows<OP, T, float, NV>
                       : (const void*)warp_rows<OP, T, bf16, NV>;
}

template <int NV>
static const void* wr_pick(KernelKey k) {
    switch (k.op) {
        case kSoftmax: return k.dtype == 0 ? (const void*)warp_rows<kSoftmax, float, float, NV>
                                           : (const void*)warp_rows<kSoftmax, bf16, float, NV>;
        case kLayerNorm: return k.dtype == 0 ? wr_param<kLayerNorm, float, NV>(k.pdtype)
                                             : wr_param<kLayerNorm, bf16, NV>(k.pdtype);
        case kRMSNorm: return k.dtype == 0 ? wr_param<kRMSNorm, float, NV>(k.pdtype)
                                           : wr_param<kRMSNorm, bf16, NV>(k.pdtype);
    }
    return nullptr;
}

const void* warp_rows_kernel(KernelKey k, int64_t nvec) {
    if (!k.vec || nvec < 1 || nvec > 32 * kWarpRowNV) return nullptr;  // whole vectors only
    const bool half = k.op != kSoftmax && nvec <= 32 * (kWarpRowNV / 2);
    return half ? wr_pick<kWarpRowNV / 2>(k) : wr_pick<kWarpRowNV>(k);
}

cudaError_t launch_warp_rows(KernelKey k, const WarpRowsArgs& a, int blocks, cudaStream_t s) {
    const int es = k.dtype == 0 ? 4 : 2;
    const void* fn = warp_rows_kernel(k, a.cols * es / 16);
    if (!fn) return cudaErrorInvalidDeviceFunction;
    WarpRowsArgs b = a;
    void* args[] = {&b};
    return cudaLaunchKernel(fn, dim3((unsigned)blocks), dim3((unsigned)kWarpRowThreads), args, 0, s);
}

}  // namespace credit
