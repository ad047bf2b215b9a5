// rowops.cuh -- the per-element arithmetic of the three operators, written
// with Blackwell's packed fp32x2 instructions (fma / add / sub / mul .f32x2)
// so that two elements cost one floating-point instruction, plus the
// per-thread statistics, the CTA-level partial and the output map h.
//
// Statistics per thread (CREDIT summary page, arXiv 2609.01864v1, "C.
// Cluster Reduction and Reuse Protocol": thread accumulation, then warp
// shuffles, then a shared-memory fold):
//   RMSNorm          sum of squares
//   LayerNorm        shifted sums around the thread's first element K:
//                    n, s1 = sum (x - K), s2 = sum (x - K)^2
//   softmax, bf16    online (m, s): running max, sum of exp relative to it
//   softmax, fp32    the max only; a second local pass over the staged slice
//                    then writes t = exp(x - m_q) back in place and sums it,
//                    so the output pass is a single multiply
#pragma once

#include "common.cuh"

namespace credit {

// ------------------------------------------------------------ packed math
// float2 pairs and the sm_100-family packed builtins (one FFMA2 / FADD2 /
// FMUL2 per two elements, round to nearest).
using F2 = float2;

__device__ __forceinline__ F2 f2(float v) { return make_float2(v, v); }
__device__ __forceinline__ F2 fma2(F2 a, F2 b, F2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ F2 add2(F2 a, F2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ F2 mul2(F2 a, F2 b) { return __fmul2_rn(a, b); }
// three-input max
__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// ----------------------------------------------------------- warp tiles
// Work over a contiguous staged range is split into warp tiles of 32 x U
// items: warp w takes tiles w, w + nwarps, ...; lane l takes items
// tile + l + 32u.  Lane offsets inside a tile are compile-time constants and
// only the one partial tile of a warp carries bounds checks.
template <int U, typename F>
__device__ __forceinline__ void for_tiles(int n, int warp, int nwarps, int lane, F f) {
    constexpr int kTile = 32 * U;
    int t = warp * kTile;
    for (; t + kTile <= n; t += nwarps * kTile) {
#pragma unroll
        for (int u = 0; u < U; ++u) f(t + lane + 32 * u);
    }
    if (t < n) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = t + lane + 32 * u;
            if (i < n) f(i);
        }
    }
}

// 16-byte vector <-> element pairs (VEC / 2 pairs)
template <typename T> struct Pairs;
template <> struct Pairs<float> {
    static constexpr int kN = 2;
    __device__ static void unpack(uint4 v, F2* p) {
        p[0] = {__uint_as_float(v.x), __uint_as_float(v.y)};
        p[1] = {__uint_as_float(v.z), __uint_as_float(v.w)};
    }
    __device__ static uint4 pack(const F2* p) {
        return make_uint4(__float_as_uint(p[0].x), __float_as_uint(p[0].y),
                          __float_as_uint(p[1].x), __float_as_uint(p[1].y));
    }
};
template <> struct Pairs<bf16> {
    static constexpr int kN = 4;
    __device__ static F2 one(uint32_t w) {
        return {__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u)};
    }
    __device__ static void unpack(uint4 v, F2* p) {
        p[0] = one(v.x); p[1] = one(v.y); p[2] = one(v.z); p[3] = one(v.w);
    }
    __device__ static uint32_t two(F2 a) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a.x, a.y);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __device__ static uint4 pack(const F2* p) {
        return make_uint4(two(p[0]), two(p[1]), two(p[2]), two(p[3]));
    }
};

// Per-column parameters of one 16-byte vector as pairs (absent = fill).
template <typename PT, int NP>
__device__ __forceinline__ void load_param_pairs(const PT* p, int64_t j0, F2* out, float fill) {
    constexpr int VEC = 2 * NP;
    if (!p) {
#pragma unroll
        for (int i = 0; i < NP; ++i) out[i] = f2(fill);
        return;
    }
    float v[VEC];
    load_params<PT, VEC>(p, j0, v);
#pragma unroll
    for (int i = 0; i < NP; ++i) out[i] = {v[2 * i], v[2 * i + 1]};
}

// ------------------------------------------------------- thread statistics
template <int OP, typename T> struct Stats;

template <typename T> struct Stats<kRMSNorm, T> {
    F2 q = {0.f, 0.f};
    __device__ __forceinline__ void add(uint4 raw) {
        F2 p[Pairs<T>::kN];
        Pairs<T>::unpack(raw, p);
#pragma unroll
        for (int i = 0; i < Pairs<T>::kN; ++i) q = fma2(p[i], p[i], q);
    }
    __device__ __forceinline__ void add1(float f) { q.x = fmaf(f, f, q.x); }
};

template <typename T> struct Stats<kLayerNorm, T> {
    F2 nK = {0.f, 0.f}, s1 = {0.f, 0.f}, s2 = {0.f, 0.f};  // nK = -K in both lanes
    float n = 0.f;
    __device__ __forceinline__ void add(uint4 raw) {
        F2 p[Pairs<T>::kN];
        Pairs<T>::unpack(raw, p);
        if (n == 0.f) nK = f2(-p[0].x);
#pragma unroll
        for (int i = 0; i < Pairs<T>::kN; ++i) {
            const F2 d = add2(p[i], nK);
            s1 = add2(s1, d);
            s2 = fma2(d, d, s2);
        }
        n += (float)(2 * Pairs<T>::kN);
    }
    __device__ __forceinline__ void add1(float f) {
        if (n == 0.f) nK = f2(-f);
        const float d = f + nK.x;
        s1.x += d;
        s2.x = fmaf(d, d, s2.x);
        n += 1.f;
    }
};

// bf16 softmax: online max and sum of exp relative to it
template <> struct Stats<kSoftmax, bf16> {
    float m = -INFINITY;
    F2 s = {0.f, 0.f};
    __device__ __forceinline__ void rebase(float vm) {
        if (vm > m) {
            const float sc = (s.x == 0.f && s.y == 0.f) ? 0.f : fast_ex2((m - vm) * kLog2e);
            s = mul2(s, f2(sc));
            m = vm;
        }
    }
    __device__ __forceinline__ void add(uint4 raw) {
        F2 p[4];
        Pairs<bf16>::unpack(raw, p);
        const float vm = fmaxf(max3(p[0].x, p[0].y, p[1].x), max3(p[1].y, p[2].x, max3(p[2].y, p[3].x, p[3].y)));
        rebase(vm);
        const F2 nm = f2(-m * kLog2e), l2 = f2(kLog2e);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const F2 a = fma2(p[i], l2, nm);
            s = add2(s, F2{fast_ex2(a.x), fast_ex2(a.y)});
        }
    }
    __device__ __forceinline__ void add1(float f) {
        rebase(f);
        s.x += fast_ex2(fmaf(f, kLog2e, -m * kLog2e));
    }
};

// fp32 softmax: the max only (the sum comes from the stash pass)
template <> struct Stats<kSoftmax, float> {
    float m = -INFINITY;
    __device__ __forceinline__ void add(uint4 raw) {
        m = max3(m, max3(__uint_as_float(raw.x), __uint_as_float(raw.y), __uint_as_float(raw.z)),
                 __uint_as_float(raw.w));
    }
    __device__ __forceinline__ void add1(float f) { m = fmaxf(m, f); }
};

// quantization: the row's absolute maximum
template <typename T> struct Stats<kQuant, T> {
    float a = 0.f;
    __device__ __forceinline__ void add(uint4 raw) {
        F2 p[Pairs<T>::kN];
        Pairs<T>::unpack(raw, p);
#pragma unroll
        for (int i = 0; i < Pairs<T>::kN; ++i) a = max3(a, fabsf(p[i].x), fabsf(p[i].y));
    }
    __device__ __forceinline__ void add1(float f) { a = fmaxf(a, fabsf(f)); }
};

// weighted standardization: weighted shifted sums around the thread's first
// element K: W = sum w, s1 = sum w (x - K), s2 = sum w (x - K)^2
template <typename T> struct Stats<kWStd, T> {
    F2 nK = {0.f, 0.f}, sw = {0.f, 0.f}, s1 = {0.f, 0.f}, s2 = {0.f, 0.f};
    bool started = false;
    __device__ __forceinline__ void add(uint4 raw, const F2* w) {
        F2 p[Pairs<T>::kN];
        Pairs<T>::unpack(raw, p);
        if (!started) { nK = f2(-p[0].x); started = true; }
#pragma unroll
        for (int i = 0; i < Pairs<T>::kN; ++i) {
            const F2 d = add2(p[i], nK);
            const F2 wd = mul2(w[i], d);
            sw = add2(sw, w[i]);
            s1 = add2(s1, wd);
            s2 = fma2(wd, d, s2);
        }
    }
    __device__ __forceinline__ void add1(float f, float w) {
        if (!started) { nK = f2(-f); started = true; }
        const float d = f + nK.x;
        sw.x += w;
        s1.x = fmaf(w, d, s1.x);
        s2.x = fmaf(w * d, d, s2.x);
    }
};

// fp32 softmax stash pass over the staged vectors [0, nvec) at `base`:
// t = exp(x - mq) written back in place (accurate expf); returns this
// thread's sum of t.  Vectors are visited in the same warp tiles as the
// output pass, so each thread re-reads exactly what it wrote.
__device__ __forceinline__ float softmax_stash(unsigned char* base, int nvec, int warp, int nwarps,
                                               int lane, float mq) {
    F2 s = {0.f, 0.f};
    for_tiles<4>(nvec, warp, nwarps, lane, [&](int v) {
        unsigned char* a = base + (size_t)v * 16;
        const uint4 raw = lds16(a);
        const F2 t0 = {expf(__uint_as_float(raw.x) - mq), expf(__uint_as_float(raw.y) - mq)};
        const F2 t1 = {expf(__uint_as_float(raw.z) - mq), expf(__uint_as_float(raw.w) - mq)};
        s = add2(s, add2(t0, t1));
        *reinterpret_cast<uint4*>(a) = make_uint4(__float_as_uint(t0.x), __float_as_uint(t0.y),
                                                  __float_as_uint(t1.x), __float_as_uint(t1.y));
    });
    return s.x + s.y;
}

// ---------------------------------------------------------- CTA partial
// The CTA's compact partial from its threads' statistics: softmax (m, s),
// LayerNorm (n, mean, M2), RMSNorm (ss).  At most two block reductions and
// no per-step division: LayerNorm reduces (n, sum n_t mean_t), then
// sum M2_t + n_t (mean_t - mean)^2 (the parallel-axis form of Chan et al.'s
// merge); softmax reduces the max, then each thread's sum rescaled to it.
// redA / redB: 2 floats per warp each.  For fp32 softmax `stash_sum` runs
// the stash pass with the CTA max and returns the thread's sum.
template <int OP, typename T, typename StashFn>
__device__ __forceinline__ void cta_partial(const Stats<OP, T>& st, float* redA, float* redB,
                                            int nwarps, int nthreads, StashFn stash_sum,
                                            float& p0, float& p1, float& p2) {
    p1 = p2 = 0.f;
    float unused = 0.f;
    if constexpr (OP == kSoftmax) {
        const float m = block_max1(st.m, redA, nwarps, nthreads);
        float s;
        if constexpr (sizeof(T) == 4) s = m == -INFINITY ? 0.f : stash_sum(m);
        else s = rescale(st.s.x + st.s.y, st.m, m);
        block_sum2(s, unused, redB, nwarps, nthreads);
        p0 = m; p1 = s;
    } else if constexpr (OP == kLayerNorm) {
        const float s1 = st.s1.x + st.s1.y, s2 = st.s2.x + st.s2.y;
        const float mt = st.n > 0.f ? s1 / st.n - st.nK.x : 0.f;
        const float m2t = st.n > 0.f ? fmaxf(s2 - s1 * (s1 / st.n), 0.f) : 0.f;
        float n = st.n, nm = st.n * mt;
        block_sum2(n, nm, redA, nwarps, nthreads);
        const float mean = n > 0.f ? nm / n : 0.f;
        const float d = mt - mean;
        float q = fmaf(st.n * d, d, m2t);
        block_sum2(q, unused, redB, nwarps, nthreads);
        p0 = n; p1 = mean; p2 = q;
    } else {
        float ss = st.q.x + st.q.y;
        block_sum2(ss, unused, redA, nwarps, nthreads);
        p0 = ss;
    }
}

// ------------------------------------------------------------ output map
// h from the combined statistics (st0, st1, st2) of a row of N columns and
// (fp32 softmax) the CTA's own max mq:
//   softmax bf16  y = 2^(x log2 e - m log2 e) / s
//   softmax fp32  y = t * (exp(mq - m) / s), t = exp(x - mq) from the stash
//   LayerNorm     y = (x r - mean r) gamma + beta,  r = 1 / sqrt(M2 / N + eps)
//   RMSNorm       y = (x r) w,                      r = 1 / sqrt(ss / N + eps)
template <int OP, typename T>
struct OutputMap {
    float c0 = 0.f, c1 = 0.f;
    __device__ __forceinline__ OutputMap() {}
    __device__ __forceinline__ OutputMap(float st0, float st1, float st2, float mq, int64_t N,
                                         float eps) {
        if constexpr (OP == kQuant) {
            c0 = st0 / 127.f;  // the row scale (IEEE division)
            c1 = quant_inv(c0);
        } else if constexpr (OP == kWStd) {
            const float r = 1.f / sqrtf(fmaxf(st0 > 0.f ? st2 / st0 : 0.f, 0.f) + eps);
            c0 = r;
            c1 = -st1 * r;
        } else if constexpr (OP == kSoftmax) {
            if constexpr (sizeof(T) == 4) { c1 = rescale(1.f, mq, st0) / st1; }
            else { c0 = -st0 * kLog2e; c1 = 1.f / st1; }
        } else if constexpr (OP == kLayerNorm) {
            const float r = 1.f / sqrtf(fmaxf(st2 / (float)N, 0.f) + eps);
            c0 = r;
            c1 = -st1 * r;
        } else {
            c0 = 1.f / sqrtf(st0 / (float)N + eps);
        }
    }
    // int8 code of x (quantization): round half to even of x / scale, clamped
    __device__ __forceinline__ int code(float x) const { return quant_code(x, c0, c1); }
    __device__ __forceinline__ F2 operator()(F2 x, F2 g, F2 b) const {
        if constexpr (OP == kWStd) {
            return fma2(x, f2(c0), f2(c1));
        } else if constexpr (OP == kSoftmax) {
            if constexpr (sizeof(T) == 4) return mul2(x, f2(c1));
            const F2 a = fma2(x, f2(kLog2e), f2(c0));
            return mul2(F2{fast_ex2(a.x), fast_ex2(a.y)}, f2(c1));
        } else if constexpr (OP == kLayerNorm) {
            return fma2(fma2(x, f2(c0), f2(c1)), g, b);
        } else {
            return mul2(mul2(x, f2(c0)), g);
        }
    }
    // the same arithmetic on one element (element path)
    __device__ __forceinline__ float one(float x, float g, float b) const {
        if constexpr (OP == kWStd) {
            return fmaf(x, c0, c1);
        } else if constexpr (OP == kSoftmax) {
            if constexpr (sizeof(T) == 4) return x * c1;
            return fast_ex2(fmaf(x, kLog2e, c0)) * c1;
        } else if constexpr (OP == kLayerNorm) {
            return fmaf(fmaf(x, c0, c1), g, b);
        } else {
            return (x * c0) * g;
        }
    }
};

// Statistics over staged 16-byte vectors [0, n) at `base`; `wp` are the
// per-column weights of those vectors (weighted standardization only).
template <int OP, typename T, typename PT = float>
__device__ __forceinline__ void stats_tiles(Stats<OP, T>& st, const unsigned char* base, int n,
                                            int warp, int nwarps, int lane,
                                            const PT* wp = nullptr) {
    if constexpr (OP == kWStd) {
        constexpr int NP = Pairs<T>::kN;
        for_tiles<4>(n, warp, nwarps, lane, [&](int v) {
            F2 w[NP];
            load_param_pairs<PT, NP>(wp, (int64_t)v * 2 * NP, w, 1.f);
            st.add(lds16(base + (size_t)v * 16), w);
        });
    } else {
        for_tiles<4>(n, warp, nwarps, lane, [&](int v) { st.add(lds16(base + (size_t)v * 16)); });
    }
}

// Statistics over [0, n) 16-byte vectors in global memory at `g` (the L2
// tail of a slice: its first read, from HBM, with the L2 policy `pol`).
// Each warp tile issues all its loads (eight per lane) before folding any.
template <int OP, typename T>
__device__ __forceinline__ void stats_global(Stats<OP, T>& st, const unsigned char* g, int n,
                                             int warp, int nwarps, int lane, uint64_t pol) {
    constexpr int U = 8, kTile = 32 * U;
    int t = warp * kTile;
    for (; t + kTile <= n; t += nwarps * kTile) {
        uint4 r[U];
#pragma unroll
        for (int u = 0; u < U; ++u) r[u] = ld_global_l2hint_v4(g + (size_t)(t + lane + 32 * u) * 16, pol);
#pragma unroll
        for (int u = 0; u < U; ++u) st.add(r[u]);
    }
    if (t < n) {
        uint4 r[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = t + lane + 32 * u;
            if (i < n) r[u] = ld_global_l2hint_v4(g + (size_t)i * 16, pol);
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (t + lane + 32 * u < n) st.add(r[u]);
    }
}

// Output granule of an operator: 4 elements for bf16 data with fp32
// parameters (so one 16-byte gamma load and one 16-byte beta load cover it),
// else one 16-byte vector of data.
template <int OP, typename T, typename PT>
struct Granule {
    static constexpr bool kHalf =
        (OP == kLayerNorm || OP == kRMSNorm) && sizeof(T) == 2 && sizeof(PT) == 4;
    static constexpr int kElems = kHalf ? 4 : 16 / (int)sizeof(T);
    static constexpr int kBytes = kElems * (int)sizeof(T);
    static constexpr int kPairs = kElems / 2;
};

// Load the parameters of one granule (kElems values, <= 16 bytes) as pairs;
// SMEM: `p` points into shared memory (a slice staged once by the caller),
// else into global memory (read-only path).
template <typename T> __device__ __forceinline__ T param_ld(const T* p, bool smem) {
    return smem ? *p : __ldg(p);
}

template <typename PT, int NP, bool SMEM = false>
__device__ __forceinline__ void granule_params(const PT* p, int q, F2* out) {
    if constexpr (sizeof(PT) == 4) {
        if constexpr (NP == 2) {
            const float4 v = param_ld(reinterpret_cast<const float4*>(p) + q, SMEM);
            out[0] = make_float2(v.x, v.y);
            out[1] = make_float2(v.z, v.w);
        } else {  // NP == 4 cannot happen for fp32 parameters (16 bytes max)
            static_assert(NP == 2, "fp32 parameters: 4 per granule");
        }
    } else {
        if constexpr (NP == 4) {
            const uint4 v = param_ld(reinterpret_cast<const uint4*>(p) + q, SMEM);
            Pairs<bf16>::unpack(v, out);
        } else {
            const uint2 v = param_ld(reinterpret_cast<const uint2*>(p) + q, SMEM);
            out[0] = Pairs<bf16>::one(v.x);
            out[1] = Pairs<bf16>::one(v.y);
        }
    }
}

// No-op progress hook of output_tiles.
struct NoRelease {
    __device__ __forceinline__ void operator()(int) const {}
};

// Apply h to the staged slice ([0, nvec) 16-byte vectors at `base`) and
// store it to `yrow`; gp / bp are the slice's parameters (null = absent).
// Each warp tile loads all its data and parameters before its first store,
// so parameter fetches overlap instead of queueing behind stores.  After
// each tile `release(v)` is told the first staged vector the warp may still
// read (the start of its next tile; nvec at the end), so a caller can hand
// back the shared memory the warp has finished with.  SMEM: gp / bp point to
// a copy of the slice's parameters in shared memory.  XG: `base` is global
// memory (the L2 tail of a slice, read a second time), loaded past L1 with
// the L2 policy `xpol`; each element is loaded before the same lane stores
// its output, so y may alias x.
template <int OP, typename T, typename PT, typename Release = NoRelease, bool SMEM = false,
          bool XG = false>
__device__ __forceinline__ void output_tiles(const OutputMap<OP, T>& h, const unsigned char* base,
                                             T* yrow, const PT* gp, const PT* bp, int nvec,
                                             int warp, int nwarps, int lane,
                                             Release release = Release(), uint64_t xpol = 0) {
    using G = Granule<OP, T, PT>;
    // granules in flight per lane: the L2 tail (XG) is latency-bound on its
    // loads, so it keeps more of them in flight than the shared-memory pass
    constexpr int kU = (OP != kSoftmax && G::kPairs == 4) ? 2 : 4;
    constexpr int U = XG ? (OP == kSoftmax ? 8 : 4) : kU, NP = G::kPairs, kTile = 32 * U;
    const int ngran = nvec * (16 / G::kBytes);
    constexpr bool kParams = OP == kLayerNorm || OP == kRMSNorm;
    const bool has_g = kParams && gp != nullptr;
    const bool has_b = kParams && bp != nullptr;

    auto tile = [&](int t, bool full) {
        uint4 raw[U];
        F2 gv[U][NP], bv[U][NP];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int q = t + lane + 32 * u;
            if (full || q < ngran) {
                if constexpr (G::kBytes == 8) {
                    uint2 w;
                    if constexpr (XG) w = ld_global_l2hint_v2(base + (size_t)q * 8, xpol);
                    else w = *reinterpret_cast<const uint2*>(base + (size_t)q * 8);
                    raw[u] = make_uint4(w.x, w.y, 0u, 0u);
                } else {
                    if constexpr (XG) raw[u] = ld_global_l2hint_v4(base + (size_t)q * 16, xpol);
                    else raw[u] = lds16(base + (size_t)q * 16);
                }
                if constexpr (kParams) {
                    if (has_g) granule_params<PT, NP, SMEM>(gp, q, gv[u]);
                    else for (int i = 0; i < NP; ++i) gv[u][i] = f2(1.f);
                    if (has_b) granule_params<PT, NP, SMEM>(bp, q, bv[u]);
                    else for (int i = 0; i < NP; ++i) bv[u][i] = f2(0.f);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int q = t + lane + 32 * u;
            if (full || q < ngran) {
                F2 p[NP];
                if constexpr (G::kBytes == 8) {
                    p[0] = Pairs<bf16>::one(raw[u].x);
                    p[1] = Pairs<bf16>::one(raw[u].y);
                } else {
                    Pairs<T>::unpack(raw[u], p);
                }
#pragma unroll
                for (int i = 0; i < NP; ++i) {
                    if constexpr (kParams) p[i] = h(p[i], gv[u][i], bv[u][i]);
                    else p[i] = h(p[i], p[i], p[i]);
                }
                if constexpr (G::kBytes == 8) {
                    __stcs(reinterpret_cast<uint2*>(yrow) + q,
                           make_uint2(Pairs<bf16>::two(p[0]), Pairs<bf16>::two(p[1])));
                } else {
                    stg16_stream(reinterpret_cast<uint4*>(yrow) + q, Pairs<T>::pack(p));
                }
            }
        }
    };
    constexpr int kGranPerVec = 16 / G::kBytes;
    int t = warp * kTile;
    for (; t + kTile <= ngran; t += nwarps * kTile) {
        tile(t, true);
        release(min(nvec, (t + nwarps * kTile) / kGranPerVec));
    }
    if (t < ngran) tile(t, false);
    release(nvec);
}

// Output of one row slice with an L2 tail, the tail written from shared
// memory: `stage` holds the first `nvec` vectors of the slice, `xtail` (global
// memory) the `ntv` vectors that follow them, which the statistics pass read
// from HBM with an evict-last policy.  A warp's first D full staged tiles,
// once written, are read by no one else, so they become the warp's private
// ring: after writing staged tile k < D, each lane copies its own vectors of
// the warp's tail tile k into its own vectors of that tile (cp.async from L2,
// evict-first, no registers held while they fly), and after writing tail
// tile j from its slot it refills the slot with tail tile j + D.  The warp
// writes its tail right after those D tiles, so that the tail's lines are
// read again soon after the statistics pass left them in L2, and its other
// staged tiles last.  Every copy is read back by the lane
// that issued it, after its own wait, so no barrier is needed; D tiles of
// every warp are in flight.  A warp with fewer than D full staged tiles
// takes a ring of D / 2 (down to two), and with fewer than two reads its
// tail tiles from global memory instead.  gp / bp point to the slice's
// first parameter; y may alias x (each tail element is copied before the
// same lane stores its output, and staged columns never overlap the tail).
template <int OP, typename T, typename PT, int D>
__device__ __forceinline__ void output_ring(const OutputMap<OP, T>& h, const unsigned char* stage,
                                            const unsigned char* xtail, T* yrow, const PT* gp,
                                            const PT* bp, int nvec, int ntv, int warp,
                                            int nwarps, int lane, uint64_t tail_pol) {
    using G = Granule<OP, T, PT>;
    static_assert(G::kBytes == 16, "the ring copies 16-byte granules");
    constexpr int U = (OP != kSoftmax && G::kPairs == 4) ? 2 : 4, NP = G::kPairs, kTile = 32 * U;
    constexpr bool kParams = OP == kLayerNorm || OP == kRMSNorm;
    const bool has_g = kParams && gp != nullptr;
    const bool has_b = kParams && bp != nullptr;
    const int stride = nwarps * kTile, t0 = warp * kTile;
    const bool ring = t0 + (D - 1) * stride + kTile <= nvec;
    if constexpr (D > 2) {
        // too few full staged tiles for this depth: a shallower ring
        if (!ring) {
            output_ring<OP, T, PT, D / 2>(h, stage, xtail, yrow, gp, bp, nvec, ntv, warp, nwarps,
                                          lane, tail_pol);
            return;
        }
    }
    const uint32_t s0 = smem_u32(stage);
    // src_t: the tile's first granule in shared memory (xg: read from the
    // tail in global memory instead); dst_t: the granule index of its output
    // and parameters within the slice; lim: the granule count at dst
    auto tile = [&](int src_t, int dst_t, int lim, bool xg) {
        const bool full = dst_t + kTile <= lim;
        uint4 raw[U];
        F2 gv[U][NP], bv[U][NP];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int q = dst_t + lane + 32 * u;
            if (full || q < lim) {
                if (xg) raw[u] = ld_global_l2hint_v4(xtail + (size_t)(q - nvec) * 16, tail_pol);
                else raw[u] = lds16(stage + (size_t)(src_t + lane + 32 * u) * 16);
                if constexpr (kParams) {
                    if (has_g) granule_params<PT, NP>(gp, q, gv[u]);
                    else for (int i = 0; i < NP; ++i) gv[u][i] = f2(1.f);
                    if (has_b) granule_params<PT, NP>(bp, q, bv[u]);
                    else for (int i = 0; i < NP; ++i) bv[u][i] = f2(0.f);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int q = dst_t + lane + 32 * u;
            if (full || q < lim) {
                F2 p[NP];
                Pairs<T>::unpack(raw[u], p);
#pragma unroll
                for (int i = 0; i < NP; ++i) {
                    if constexpr (kParams) p[i] = h(p[i], gv[u][i], bv[u][i]);
                    else p[i] = h(p[i], p[i], p[i]);
                }
                stg16_stream(reinterpret_cast<uint4*>(yrow) + q, Pairs<T>::pack(p));
            }
        }
    };
    // tail tile k of this warp into ring slot k % D (one commit group, empty
    // past the tail, so that the groups stay counted)
    auto prefetch = [&](int k) {
        const int tt = t0 + k * stride, ts = t0 + (k % D) * stride;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int q = tt + lane + 32 * u;
            if (q < ntv)
                cp_async16(s0 + (uint32_t)(ts + lane + 32 * u) * 16u, xtail + (size_t)q * 16,
                           tail_pol);
        }
        cp_async_commit();
    };
    const int lim = nvec + ntv;
    int t = t0;
    if (ring) {
        // the first D staged tiles (full), each freeing a ring slot; then the
        // tail, so that its lines are read again soon after the statistics
        // pass left them in L2; then the rest of the staged tiles
        for (int k = 0; k < D; ++k, t += stride) {
            tile(t, t, nvec, false);
            prefetch(k);
        }
        // D groups were committed above and one more per tail tile, so tail
        // tile j's group is complete once at most D - 1 are pending
        for (int j = 0; t0 + j * stride < ntv; ++j) {
            cp_async_wait<D - 1>();
            const int tt = t0 + j * stride;
            tile(t0 + (j % D) * stride, nvec + tt, lim, false);
            prefetch(j + D);
        }
        cp_async_wait<0>();
    } else {
        // the tail first, from global memory
        for (int tt = t0; tt < ntv; tt += stride) tile(0, nvec + tt, lim, true);
    }
    for (; t + kTile <= nvec; t += stride) tile(t, t, nvec, false);
    if (t < nvec) tile(t, t, nvec, false);
}

}  // namespace credit

namespace credit {

// ----------------------------------------------------- multi-row tiles
// Block-wide sums / maxima of N values per thread (named barrier 1 over the
// first `nthreads` threads); every participating thread returns the folded
// values.  `red` holds N floats per warp and must not be read by any thread
// from an earlier use.
template <int N, bool kMax>
__device__ __forceinline__ void block_reduce_n(float (&x)[N], float* red, int nwarps, int nthreads) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const float y = __shfl_xor_sync(0xffffffffu, x[i], o);
            x[i] = kMax ? fmaxf(x[i], y) : x[i] + y;
        }
    }
    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < N; ++i) red[N * warp + i] = x[i];
    }
    named_sync(nthreads);
#pragma unroll
    for (int i = 0; i < N; ++i) x[i] = kMax ? -INFINITY : 0.f;
    for (int w = 0; w < nwarps; ++w) {
#pragma unroll
        for (int i = 0; i < N; ++i) x[i] = kMax ? fmaxf(x[i], red[N * w + i]) : x[i] + red[N * w + i];
    }
}

// The CTA partials of R rows at once (see cta_partial): two block reductions
// of R or 2R values in total instead of two per row.  stash_sum(i, mq) runs
// the fp32 softmax stash pass of row i.  redA / redB: 2R floats per warp.
template <int OP, typename T, int R, typename StashFn>
__device__ __forceinline__ void cta_partial_rows(const Stats<OP, T> (&st)[R], float* redA,
                                                 float* redB, int nwarps, int nthreads,
                                                 StashFn stash_sum, float (&p)[R][3]) {
    if constexpr (OP == kQuant) {
        float a[R];
#pragma unroll
        for (int i = 0; i < R; ++i) a[i] = st[i].a;
        block_reduce_n<R, true>(a, redA, nwarps, nthreads);
#pragma unroll
        for (int i = 0; i < R; ++i) { p[i][0] = a[i]; p[i][1] = p[i][2] = 0.f; }
    } else if constexpr (OP == kWStd) {
        float a[2 * R], mt[R], m2t[R], wt[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const float W = st[i].sw.x + st[i].sw.y;
            const float s1 = st[i].s1.x + st[i].s1.y, s2 = st[i].s2.x + st[i].s2.y;
            wt[i] = W;
            mt[i] = W > 0.f ? s1 / W - st[i].nK.x : 0.f;
            m2t[i] = W > 0.f ? fmaxf(s2 - s1 * (s1 / W), 0.f) : 0.f;
            a[2 * i] = W;
            a[2 * i + 1] = W * mt[i];
        }
        block_reduce_n<2 * R, false>(a, redA, nwarps, nthreads);
        float q[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const float mean = a[2 * i] > 0.f ? a[2 * i + 1] / a[2 * i] : 0.f;
            const float d = mt[i] - mean;
            q[i] = fmaf(wt[i] * d, d, m2t[i]);
            p[i][0] = a[2 * i];
            p[i][1] = mean;
        }
        block_reduce_n<R, false>(q, redB, nwarps, nthreads);
#pragma unroll
        for (int i = 0; i < R; ++i) p[i][2] = q[i];
    } else if constexpr (OP == kSoftmax) {
        float m[R];
#pragma unroll
        for (int i = 0; i < R; ++i) m[i] = st[i].m;
        block_reduce_n<R, true>(m, redA, nwarps, nthreads);
        float s[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            if constexpr (sizeof(T) == 4) s[i] = m[i] == -INFINITY ? 0.f : stash_sum(i, m[i]);
            else s[i] = rescale(st[i].s.x + st[i].s.y, st[i].m, m[i]);
        }
        block_reduce_n<R, false>(s, redB, nwarps, nthreads);
#pragma unroll
        for (int i = 0; i < R; ++i) { p[i][0] = m[i]; p[i][1] = s[i]; p[i][2] = 0.f; }
    } else if constexpr (OP == kLayerNorm) {
        float a[2 * R], mt[R], m2t[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const float s1 = st[i].s1.x + st[i].s1.y, s2 = st[i].s2.x + st[i].s2.y, nn = st[i].n;
            mt[i] = nn > 0.f ? s1 / nn - st[i].nK.x : 0.f;
            m2t[i] = nn > 0.f ? fmaxf(s2 - s1 * (s1 / nn), 0.f) : 0.f;
            a[2 * i] = nn;
            a[2 * i + 1] = nn * mt[i];
        }
        block_reduce_n<2 * R, false>(a, redA, nwarps, nthreads);
        float q[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const float mean = a[2 * i] > 0.f ? a[2 * i + 1] / a[2 * i] : 0.f;
            const float d = mt[i] - mean;
            q[i] = fmaf(st[i].n * d, d, m2t[i]);
            p[i][0] = a[2 * i];
            p[i][1] = mean;
        }
        block_reduce_n<R, false>(q, redB, nwarps, nthreads);
#pragma unroll
        for (int i = 0; i < R; ++i) p[i][2] = q[i];
    } else {
        float q[R];
#pragma unroll
        for (int i = 0; i < R; ++i) q[i] = st[i].q.x + st[i].q.y;
        block_reduce_n<R, false>(q, redA, nwarps, nthreads);
#pragma unroll
        for (int i = 0; i < R; ++i) { p[i][0] = q[i]; p[i][1] = p[i][2] = 0.f; }
    }
}

// Output of one row with parameters, software-pipelined: a warp's next tile
// of parameters is requested before the current tile is computed and stored,
// so their L2 latency overlaps the work instead of stalling each tile (the
// parameter vectors are re-read by every row, from L2).  Two register sets
// alternate; tiles are U granules per lane.
template <int OP, typename T, typename PT, int U>
__device__ __forceinline__ void output_tiles_pipelined(const OutputMap<OP, T>& h,
                                                       const unsigned char* base, T* yrow,
                                                       const PT* gp, const PT* bp, int nvec,
                                                       int warp, int nwarps, int lane) {
    using G = Granule<OP, T, PT>;
    constexpr int NP = G::kPairs, kTile = 32 * U;
    const int ngran = nvec * (16 / G::kBytes);
    const int stride = nwarps * kTile;
    const bool has_g = gp != nullptr, has_b = bp != nullptr;

    auto load = [&](int t, F2 (&gv)[U][NP], F2 (&bv)[U][NP]) {
        const bool full = t + kTile <= ngran;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int q = t + lane + 32 * u;
            if (full || q < ngran) {
                if (has_g) granule_params<PT, NP>(gp, q, gv[u]);
                if (has_b) granule_params<PT, NP>(bp, q, bv[u]);
            }
        }
    };
    auto apply = [&](int t, const F2 (&gv)[U][NP], const F2 (&bv)[U][NP]) {
        const bool full = t + kTile <= ngran;
        uint4 raw[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int q = t + lane + 32 * u;
            if (full || q < ngran) {
                if constexpr (G::kBytes == 8) {
                    const uint2 w = *reinterpret_cast<const uint2*>(base + (size_t)q * 8);
                    raw[u] = make_uint4(w.x, w.y, 0u, 0u);
                } else {
                    raw[u] = lds16(base + (size_t)q * 16);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int q = t + lane + 32 * u;
            if (full || q < ngran) {
                F2 p[NP];
                if constexpr (G::kBytes == 8) {
                    p[0] = Pairs<bf16>::one(raw[u].x);
                    p[1] = Pairs<bf16>::one(raw[u].y);
                } else {
                    Pairs<T>::unpack(raw[u], p);
                }
#pragma unroll
                for (int i = 0; i < NP; ++i) p[i] = h(p[i], gv[u][i], bv[u][i]);
                if constexpr (G::kBytes == 8) {
                    __stcs(reinterpret_cast<uint2*>(yrow) + q,
                           make_uint2(Pairs<bf16>::two(p[0]), Pairs<bf16>::two(p[1])));
                } else {
                    stg16_stream(reinterpret_cast<uint4*>(yrow) + q, Pairs<T>::pack(p));
                }
            }
        }
    };
    F2 ga[U][NP], ba[U][NP], gb[U][NP], bb[U][NP];
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            ga[u][i] = gb[u][i] = f2(1.f);
            ba[u][i] = bb[u][i] = f2(0.f);
        }
    }
    int t = warp * kTile;
    if (t < ngran) load(t, ga, ba);
    while (t < ngran) {
        const int t1 = t + stride;
        if (t1 < ngran) load(t1, gb, bb);
        apply(t, ga, ba);
        if (t1 >= ngran) break;
        const int t2 = t1 + stride;
        if (t2 < ngran) load(t2, ga, ba);
        apply(t1, gb, bb);
        t = t2;
    }
}

// Output of R rows that share a column slice: each granule's parameters are
// loaded once and applied to all live rows (row i staged at base + i * pitch,
// written to yrow[i]); the first `rows` <= R rows are live.  XG: the rows are
// in global memory (the L2 tails of R rows, `pitch` bytes apart), loaded past
// L1 with the L2 policy `xpol`, each element before its lane stores it.
template <int OP, typename T, typename PT, int R, bool XG = false>
__device__ __forceinline__ void output_tiles_rows(const OutputMap<OP, T> (&h)[R],
                                                  const unsigned char* base, int64_t pitch,
                                                  T* const (&yrow)[R], int rows, const PT* gp,
                                                  const PT* bp, int nvec, int warp, int nwarps,
                                                  int lane, uint64_t xpol = 0) {
    using G = Granule<OP, T, PT>;
    // granules in flight per thread: 4, halved when a granule carries 8
    // parameters, divided among the rows (twice as many for an L2 tail,
    // whose loads are latency-bound)
    constexpr int kBase = ((OP != kSoftmax && G::kPairs == 4) ? 2 : 4) * (XG ? 2 : 1);
    constexpr int U = kBase / R > 0 ? kBase / R : 1, NP = G::kPairs, kTile = 32 * U;
    const int ngran = nvec * (16 / G::kBytes);
    constexpr bool kParams = OP == kLayerNorm || OP == kRMSNorm;
    const bool has_g = kParams && gp != nullptr;
    const bool has_b = kParams && bp != nullptr;

    auto tile = [&](int t, bool full) {
        uint4 raw[U][R];
        F2 gv[U][NP], bv[U][NP];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int q = t + lane + 32 * u;
            if (full || q < ngran) {
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    if (i < rows) {
                        const unsigned char* b = base + (size_t)i * pitch;
                        if constexpr (G::kBytes == 8) {
                            uint2 w;
                            if constexpr (XG) w = ld_global_l2hint_v2(b + (size_t)q * 8, xpol);
                            else w = *reinterpret_cast<const uint2*>(b + (size_t)q * 8);
                            raw[u][i] = make_uint4(w.x, w.y, 0u, 0u);
                        } else {
                            if constexpr (XG) raw[u][i] = ld_global_l2hint_v4(b + (size_t)q * 16, xpol);
                            else raw[u][i] = lds16(b + (size_t)q * 16);
                        }
                    }
                }
                if constexpr (kParams) {
                    if (has_g) granule_params<PT, NP>(gp, q, gv[u]);
                    else for (int j = 0; j < NP; ++j) gv[u][j] = f2(1.f);
                    if (has_b) granule_params<PT, NP>(bp, q, bv[u]);
                    else for (int j = 0; j < NP; ++j) bv[u][j] = f2(0.f);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int q = t + lane + 32 * u;
            if (full || q < ngran) {
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    if (i < rows) {
                        F2 pp[NP];
                        if constexpr (G::kBytes == 8) {
                            pp[0] = Pairs<bf16>::one(raw[u][i].x);
                            pp[1] = Pairs<bf16>::one(raw[u][i].y);
                        } else {
                            Pairs<T>::unpack(raw[u][i], pp);
                        }
#pragma unroll
                        for (int j = 0; j < NP; ++j) {
                            if constexpr (kParams) pp[j] = h[i](pp[j], gv[u][j], bv[u][j]);
                            else pp[j] = h[i](pp[j], pp[j], pp[j]);
                        }
                        if constexpr (G::kBytes == 8) {
                            __stcs(reinterpret_cast<uint2*>(yrow[i]) + q,
                                   make_uint2(Pairs<bf16>::two(pp[0]), Pairs<bf16>::two(pp[1])));
                        } else {
                            stg16_stream(reinterpret_cast<uint4*>(yrow[i]) + q, Pairs<T>::pack(pp));
                        }
                    }
                }
            }
        }
    };
    int t = warp * kTile;
    for (; t + kTile <= ngran; t += nwarps * kTile) tile(t, true);
    if (t < ngran) tile(t, false);
}

}  // namespace credit

namespace credit {

// Quantization output of R rows: each staged 16-byte vector becomes VEC int8
// codes (4 bytes for fp32 input, 8 for bf16), stored with one streaming
// store per vector.
template <typename T, int R>
__device__ __forceinline__ void output_quant_rows(const OutputMap<kQuant, T> (&h)[R],
                                                  const unsigned char* base, int pitch,
                                                  int8_t* const (&qrow)[R], int rows, int nvec,
                                                  int warp, int nwarps, int lane) {
    constexpr int NP = Pairs<T>::kN;
    for_tiles<4>(nvec, warp, nwarps, lane, [&](int v) {
#pragma unroll
        for (int i = 0; i < R; ++i) {
            if (i < rows) {
                F2 p[NP];
                Pairs<T>::unpack(lds16(base + (size_t)i * pitch + (size_t)v * 16), p);
                float xf[2 * NP];
#pragma unroll
                for (int k = 0; k < NP; ++k) { xf[2 * k] = p[k].x; xf[2 * k + 1] = p[k].y; }
                uint32_t w[NP / 2];
                quant_codes<2 * NP>(xf, h[i].c0, h[i].c1, w);
                if constexpr (NP == 2) __stcs(reinterpret_cast<unsigned int*>(qrow[i]) + v, w[0]);
                else __stcs(reinterpret_cast<uint2*>(qrow[i]) + v, make_uint2(w[0], w[1]));
            }
        }
    });
}

}  // namespace credit
