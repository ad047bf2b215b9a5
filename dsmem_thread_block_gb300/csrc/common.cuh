// common.cuh -- element traits, per-operator statistics and CTA-level
// reductions shared by the clustered and the two-pass kernels.
//
// Operators (CREDIT summary page, arXiv 2609.01864v1, "B. Reduction-Reuse
// Transformation": per-element inputs feed scalar statistics, then an
// elementwise h writes every output):
//   softmax   partial (m, s):      m = max x, s = sum exp(x - m)
//             combine:             m = max m_q, s = sum s_q exp(m_q - m)
//             h:                   y = exp(x - m) / s
//   LayerNorm partial (n, mu, M2): count, mean, sum of squared deviations
//             combine (Chan et al.): d = mu_b - mu_a, n = n_a + n_b,
//                                    mu = mu_a + d n_b / n,
//                                    M2 = M2_a + M2_b + d^2 n_a n_b / n
//             h:                   y = (x - mu) / sqrt(M2 / N + eps) g + b
//   RMSNorm   partial (ss):        sum x^2;  combine: sum
//             h:                   y = x / sqrt(ss / N + eps) w
// Partials are fp32; they are combined in rank order so every CTA of a
// cluster rebuilds bit-identical statistics.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace credit {

// Operators.  kQuant: row absmax -> scale -> int8 codes; kWStd: weighted
// standardization with per-column weights (the weighted counterpart of
// LayerNorm without the affine step).
enum Op : int { kSoftmax = 0, kLayerNorm = 1, kRMSNorm = 2, kQuant = 3, kWStd = 4, kPearson = 5 };

// LayerNorm-like statistics (count or weight, mean, M2).
__host__ __device__ constexpr bool norm_like(int op) { return op == kLayerNorm || op == kWStd; }

constexpr int kMaxCluster = 16;   // non-portable cluster size limit
constexpr int kMaxThreads = 512;         // two-pass kernels
constexpr int kClusterMaxThreads = 256;  // one-row-per-cluster kernel (three CTAs per SM)
constexpr int kMaxWarps = kMaxThreads / 32;
constexpr int kMaxChunks = 16;    // mbarriers per CTA for the staged slice
constexpr int kSlotStride = 4;    // floats per pushed partial (16 bytes)

// Device error word bits.
constexpr unsigned kErrTimeout = 1u;
constexpr unsigned kErrBounds = 2u;  // checked build: an index check failed

// Bounded waits give up after this long (a second or so).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

using bf16 = __nv_bfloat16;

// ---------------------------------------------------------- element traits
template <typename T> struct Elem;
template <> struct Elem<float> {
    static constexpr int kVec = 4;  // elements per 16-byte vector
    __device__ static float to_f(float v) { return v; }
    __device__ static float from_f(float v) { return v; }
    __device__ static void unpack(uint4 v, float* f) {
        f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
    }
    __device__ static uint4 pack(const float* f) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                          __float_as_uint(f[2]), __float_as_uint(f[3]));
    }
};
template <> struct Elem<bf16> {
    static constexpr int kVec = 8;
    __device__ static float to_f(bf16 v) { return __bfloat162float(v); }
    __device__ static bf16 from_f(float v) { return __float2bfloat16_rn(v); }
    __device__ static float lo(uint32_t w) { return __uint_as_float(w << 16); }
    __device__ static float hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
    __device__ static void unpack(uint4 v, float* f) {
        f[0] = lo(v.x); f[1] = hi(v.x); f[2] = lo(v.y); f[3] = hi(v.y);
        f[4] = lo(v.z); f[5] = hi(v.z); f[6] = lo(v.w); f[7] = hi(v.w);
    }
    __device__ static uint32_t pack2(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __device__ static uint4 pack(const float* f) {
        return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]),
                          pack2(f[4], f[5]), pack2(f[6], f[7]));
    }
};

// Load VEC per-column parameters starting at column j0 (j0 % VEC == 0, the
// vector 16-byte aligned when PT is the element type, 8-byte otherwise).
template <typename PT, int VEC>
__device__ __forceinline__ void load_params(const PT* p, int64_t j0, float* out) {
    static_assert(VEC == 4 || VEC == 8, "4 or 8 parameters per load");
    if constexpr (sizeof(PT) == 4) {
        const float4* q = reinterpret_cast<const float4*>(p + j0);
#pragma unroll
        for (int k = 0; k < VEC / 4; ++k) {
            float4 v = __ldg(q + k);
            out[4 * k] = v.x; out[4 * k + 1] = v.y;
            out[4 * k + 2] = v.z; out[4 * k + 3] = v.w;
        }
    } else {
        if constexpr (VEC == 8) {
            uint4 v = __ldg(reinterpret_cast<const uint4*>(p + j0));
            Elem<bf16>::unpack(v, out);
        } else {
            uint2 v = __ldg(reinterpret_cast<const uint2*>(p + j0));
            out[0] = Elem<bf16>::lo(v.x); out[1] = Elem<bf16>::hi(v.x);
            out[2] = Elem<bf16>::lo(v.y); out[3] = Elem<bf16>::hi(v.y);
        }
    }
}

template <typename PT>
__device__ __forceinline__ float load_param1(const PT* p, int64_t j) {
    if constexpr (sizeof(PT) == 4) return __ldg(reinterpret_cast<const float*>(p) + j);
    else return __bfloat162float(p[j]);
}

// ------------------------------------------------------------ exponentials
constexpr float kLog2e = 1.4426950408889634f;

// fp32 outputs use CUDA's expf (max 2 ulp); bf16 outputs use the hardware
// base-2 exponential on a pre-scaled argument, ample for a 2^-7 tolerance.
template <typename T>
__device__ __forceinline__ float exp_shift(float x, float m, float m_log2e) {
    if constexpr (sizeof(T) == 4) {
        return expf(x - m);
    } else {
        return fast_ex2(fmaf(x, kLog2e, -m_log2e));
    }
}

// ---------------------------------------------------------- statistics
struct SoftmaxPart { float m, s; };
struct NormPart { float n, mu, m2; };

// exp(a - b) * s, with s == 0 -> 0 even when a == b == -inf.
__device__ __forceinline__ float rescale(float s, float a, float b) {
    return s == 0.f ? 0.f : s * expf(a - b);
}

__device__ __forceinline__ SoftmaxPart softmax_merge(SoftmaxPart a, SoftmaxPart b) {
    float m = fmaxf(a.m, b.m);
    return {m, rescale(a.s, a.m, m) + rescale(b.s, b.m, m)};
}

__device__ __forceinline__ NormPart chan_merge(NormPart a, NormPart b) {
    if (b.n == 0.f) return a;
    if (a.n == 0.f) return b;
    float n = a.n + b.n;
    float d = b.mu - a.mu;
    float f = b.n / n;
    return {n, fmaf(d, f, a.mu), a.m2 + b.m2 + d * d * a.n * f};
}

// ------------------------------------------------------ CTA reductions
// Every thread returns the same value: lane 0 of each warp publishes its
// warp's result and every thread folds the per-warp values in warp order.
// `buf` alternates between two scratch arrays so back-to-back reductions
// need one __syncthreads each.
template <typename F>
__device__ __forceinline__ float warp_allreduce(float v, F f) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = f(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

struct SumOp { __device__ float operator()(float a, float b) const { return a + b; } };
struct MaxOp { __device__ float operator()(float a, float b) const { return fmaxf(a, b); } };

template <typename F>
__device__ __forceinline__ float block_allreduce(float v, float* buf, F f, float init) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nw = blockDim.x >> 5;
    v = warp_allreduce(v, f);
    if (lane == 0) buf[warp] = v;
    __syncthreads();
    float r = init;
    for (int w = 0; w < nw; ++w) r = f(r, buf[w]);
    return r;
}

// ---------------------------------------------------------- int8 codes
// Quantization code of x for the row scale s: round-half-even of the IEEE
// single quotient fl(x / s), clamped to +-127 -- without a division per
// element.  q = x * fl(1 / s) differs from fl(x / s) by at most 3 * 2^-24 |x/s|
// (< 2^-14 for |x / s| <= 128), so rint(q) is the code unless q lies within
// 2^-14 of a half-integer b.  There the exact residual x - b s, computed by
// one fused multiply-add (exact, since x and b s agree to within s 2^-13 and
// b carries 9 significant bits), places fl(x / s) against b: above or below
// by more than half the float spacing on that side of b, or equal to b
// (ties to even) -- the exact-remainder technique for correctly rounded
// quotients (Markstein; Boldo and Muller on the exactness of FMA
// remainders).  Scales outside [2^-90, 2^100], where those products could
// leave the normal range, use the division.
__device__ __forceinline__ float quant_inv(float s) {
    return (s >= 0x1p-90f && s <= 0x1p+100f) ? 1.f / s : 0.f;  // 0: divide per element
}

static __device__ __noinline__ float quant_near_half(float x, float s, float k, float d) {
    const float b = k + (d > 0.f ? 0.5f : -0.5f);  // the half-integer next to q (exact)
    const float rho = fmaf(-b, s, x);               // x - b s, exact
    const float away = b > 0.f ? rho : -rho;        // > 0: |x / s| beyond |b|
    const float ab = fabsf(b);
    float h_away, h_toward;                         // half the float spacing beside b
    if (ab == 0.5f) {
        h_away = 0x1p-25f;
        h_toward = 0x1p-26f;
    } else {
        h_away = h_toward = __int_as_float(__float_as_int(ab) & 0x7f800000) * 0x1p-24f;
    }
    const float out = b > 0.f ? 0.5f : -0.5f;
    if (away > s * h_away) return b + out;           // fl(x / s) beyond b
    if (away < -(s * h_toward)) return b - out;      // fl(x / s) short of b
    return rintf(b);                                 // fl(x / s) == b: ties to even
}

// The codes of N values at once, packed four to a 32-bit word (byte e of
// word e / 4): the reciprocal path for all of them and a single branch to the
// exact resolution when any quotient lies near a half-integer.
template <int N>
__device__ __forceinline__ void quant_codes(const float (&x)[N], float s, float inv,
                                            uint32_t (&w)[N / 4]) {
    constexpr float kNear = 0.5f - 0x1p-14f;
    float c[N];
    if (inv != 0.f) {
        float d[N];
        bool near = false;
#pragma unroll
        for (int e = 0; e < N; ++e) {
            const float q = x[e] * inv;
            c[e] = rintf(q);
            d[e] = q - c[e];
            near |= fabsf(d[e]) >= kNear;
        }
        if (near) {
#pragma unroll
            for (int e = 0; e < N; ++e)
                if (fabsf(d[e]) >= kNear) c[e] = quant_near_half(x[e], s, c[e], d[e]);
        }
    } else {
#pragma unroll
        for (int e = 0; e < N; ++e) c[e] = s == 0.f ? 0.f : rintf(__fdiv_rn(x[e], s));
    }
    int v[N];
#pragma unroll
    for (int e = 0; e < N; ++e) v[e] = max(-127, min(127, __float2int_rn(c[e])));
#pragma unroll
    for (int k = 0; k < N / 4; ++k) {
        const uint32_t lo = __byte_perm((uint32_t)v[4 * k], (uint32_t)v[4 * k + 1], 0x0040);
        const uint32_t hi = __byte_perm((uint32_t)v[4 * k + 2], (uint32_t)v[4 * k + 3], 0x0040);
        w[k] = __byte_perm(lo, hi, 0x5410);
    }
}

__device__ __forceinline__ int quant_code(float x, float s, float inv) {
    if (s == 0.f) return 0;
    float c;
    if (inv == 0.f) {
        c = rintf(__fdiv_rn(x, s));
    } else {
        const float q = x * inv;
        c = rintf(q);
        const float d = q - c;
        if (fabsf(d) >= 0.5f - 0x1p-14f) c = quant_near_half(x, s, c, d);
    }
    return max(-127, min(127, __float2int_rn(c)));
}

// Bounded mbarrier wait: spins on try_wait; after kWaitLimitNs sets the
// device error word and returns false (the caller carries on so that every
// cluster barrier is still reached).
__device__ __forceinline__ bool mbar_wait_limited(uint32_t bar, uint32_t parity, unsigned* err,
                                                  uint64_t limit_ns) {
    for (int i = 0; i < 256; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > limit_ns) {
            atomicOr(err, kErrTimeout);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned* err) {
    return mbar_wait_limited(bar, parity, err, kWaitLimitNs);
}

// ------------------------------------------------------------- checked build
// Index checks of the checked build (-DCREDIT_DEBUG): a failed check records
// kErrBounds in the device error word and the caller skips the access.  In
// the regular build every check is a compile-time true.
__device__ __forceinline__ bool in_bounds(bool ok, unsigned* err) {
#ifdef CREDIT_DEBUG
    if (!ok) atomicOr(err, kErrBounds);
    return ok;
#else
    (void)ok;
    (void)err;
    return true;
#endif
}

// Checked build: the combined statistics every CTA rebuilt for a row, so a
// test can see that all P CTAs of a cluster hold bit-identical values (the
// premise of the replicated push: "C. Cluster Reduction and Reuse Protocol",
// All-Gather Trade-off).  Rows [0, kDbgStatsRows) of a launch, one record of
// kDbgStatsWidth floats per (row, rank): the statistics, then P in the last.
constexpr int kDbgStatsRows = 64;
constexpr int kDbgStatsWidth = 8;

__device__ __forceinline__ void debug_row_stats(float* buf, int64_t row, uint32_t rank,
                                                uint32_t P, const float* v, int nv) {
#ifdef CREDIT_DEBUG
    if (buf && row >= 0 && row < kDbgStatsRows && rank < (uint32_t)kMaxCluster) {
        float* d = buf + ((size_t)row * kMaxCluster + rank) * kDbgStatsWidth;
        for (int i = 0; i < nv && i < kDbgStatsWidth - 1; ++i) d[i] = v[i];
        d[kDbgStatsWidth - 1] = (float)P;
    }
#else
    (void)buf; (void)row; (void)rank; (void)P; (void)v; (void)nv;
#endif
}

// Dynamic shared memory of the running launch, bytes.
__device__ __forceinline__ uint32_t dyn_smem_bytes() {
    uint32_t r;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(r));
    return r;
}

// Does a CTA's staged layout fit its launch?  `end` is one past the highest
// byte it stages into dynamic shared memory, `chunks` the chunk mbarriers (or
// ring slots) it needs of `max_chunks`.  A CTA whose layout does not fit
// stages nothing (its slice counts as empty) but still takes part in every
// exchange and cluster barrier, so its peers are not left waiting forever.
__device__ __forceinline__ bool layout_fits(uint64_t end, int64_t chunks, int max_chunks,
                                            unsigned* err) {
#ifdef CREDIT_DEBUG
    return in_bounds(end <= dyn_smem_bytes() && chunks <= max_chunks, err);
#else
    (void)end;
    (void)chunks;
    (void)max_chunks;
    (void)err;
    return true;
#endif
}

}  // namespace credit

namespace credit {

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

// Named barrier `id` among `nthreads` threads (a multiple of 32).
__device__ __forceinline__ void named_sync_id(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}

// Barrier among the first `nthreads` threads of the CTA (named barrier 1).
__device__ __forceinline__ void named_sync(int nthreads) {
    asm volatile("bar.sync 1, %0;" :: "r"(nthreads) : "memory");
}

// Fold the P pushed partials (stride kSlotStride floats) in rank order into
// the row statistics (st0, st1, st2); identical in every CTA of the cluster.
//   softmax:   m = max m_q, s = sum s_q exp(m_q - m)
//   LayerNorm: Chan et al.'s combination in its all-at-once (parallel-axis)
//              form: n = sum n_q, mean = sum n_q mean_q / n,
//              M2 = sum (M2_q + n_q (mean_q - mean)^2)
//   RMSNorm:   ss = sum ss_q
//   quantize:  amax = max amax_q;  weighted standardization: as LayerNorm
//              with weight sums in place of counts
template <int OP>
__device__ __forceinline__ void combine_slots(const float* sl, uint32_t P, float& st0,
                                              float& st1, float& st2);

// The same fold over partials `stride` floats apart (several rows' partials
// interleaved per source CTA).
template <int OP>
__device__ __forceinline__ void combine_slots_strided(const float* sl, uint32_t P, int stride,
                                                      float& st0, float& st1, float& st2) {
    if constexpr (OP == kQuant) {
        float m = 0.f;
        for (uint32_t q = 0; q < P; ++q) m = fmaxf(m, sl[q * stride]);
        st0 = m; st1 = st2 = 0.f;
    } else if constexpr (OP == kSoftmax) {
        float m = -INFINITY;
        for (uint32_t q = 0; q < P; ++q) m = fmaxf(m, sl[q * stride]);
        float s = 0.f;
        for (uint32_t q = 0; q < P; ++q) s += rescale(sl[q * stride + 1], sl[q * stride], m);
        st0 = m; st1 = s; st2 = 0.f;
    } else if constexpr (norm_like(OP)) {
        float n = 0.f, nm = 0.f;
        for (uint32_t q = 0; q < P; ++q) {
            n += sl[q * stride];
            nm = fmaf(sl[q * stride], sl[q * stride + 1], nm);
        }
        const float mean = n > 0.f ? nm / n : 0.f;
        float m2 = 0.f;
        for (uint32_t q = 0; q < P; ++q) {
            const float d = sl[q * stride + 1] - mean;
            m2 += fmaf(sl[q * stride] * d, d, sl[q * stride + 2]);
        }
        st0 = n; st1 = mean; st2 = m2;
    } else {
        float ss = 0.f;
        for (uint32_t q = 0; q < P; ++q) ss += sl[q * stride];
        st0 = ss; st1 = st2 = 0.f;
    }
}

template <int OP>
__device__ __forceinline__ void combine_slots(const float* sl, uint32_t P, float& st0,
                                              float& st1, float& st2) {
    if constexpr (OP == kQuant) {
        float m = 0.f;
        for (uint32_t q = 0; q < P; ++q) m = fmaxf(m, sl[q * kSlotStride]);
        st0 = m; st1 = st2 = 0.f;
    } else if constexpr (OP == kSoftmax) {
        float m = -INFINITY;
        for (uint32_t q = 0; q < P; ++q) m = fmaxf(m, sl[q * kSlotStride]);
        float s = 0.f;
        for (uint32_t q = 0; q < P; ++q)
            s += rescale(sl[q * kSlotStride + 1], sl[q * kSlotStride], m);
        st0 = m; st1 = s; st2 = 0.f;
    } else if constexpr (norm_like(OP)) {
        float n = 0.f, nm = 0.f;
        for (uint32_t q = 0; q < P; ++q) {
            n += sl[q * kSlotStride];
            nm = fmaf(sl[q * kSlotStride], sl[q * kSlotStride + 1], nm);
        }
        const float mean = n > 0.f ? nm / n : 0.f;
        float m2 = 0.f;
        for (uint32_t q = 0; q < P; ++q) {
            const float d = sl[q * kSlotStride + 1] - mean;
            m2 += fmaf(sl[q * kSlotStride] * d, d, sl[q * kSlotStride + 2]);
        }
        st0 = n; st1 = mean; st2 = m2;
    } else {
        float ss = 0.f;
        for (uint32_t q = 0; q < P; ++q) ss += sl[q * kSlotStride];
        st0 = ss; st1 = st2 = 0.f;
    }
}

// Block-wide reductions over the first `nthreads` threads (named barrier 1);
// every participating thread returns the same value (lane 0 of each warp
// publishes, every thread folds the warps in order).  `red` needs
// 2 floats per warp and must not be read by any thread from an earlier use.
__device__ __forceinline__ void block_sum2(float& x, float& y, float* red, int nwarps,
                                           int nthreads) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        x += __shfl_xor_sync(0xffffffffu, x, o);
        y += __shfl_xor_sync(0xffffffffu, y, o);
    }
    if (lane == 0) { red[2 * warp] = x; red[2 * warp + 1] = y; }
    named_sync(nthreads);
    x = 0.f; y = 0.f;
    for (int w = 0; w < nwarps; ++w) { x += red[2 * w]; y += red[2 * w + 1]; }
}

__device__ __forceinline__ float block_max1(float x, float* red, int nwarps, int nthreads) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    if (lane == 0) red[2 * warp] = x;
    named_sync(nthreads);
    x = -INFINITY;
    for (int w = 0; w < nwarps; ++w) x = fmaxf(x, red[2 * w]);
    return x;
}

// 16-byte shared-memory load the compiler can schedule (and order against
// the barriers, which are asm volatile with memory clobbers).
__device__ __forceinline__ uint4 lds16(const unsigned char* p) {
    return *reinterpret_cast<const uint4*>(p);
}

// 16-byte streaming global store (evict-first: the output is not re-read).
__device__ __forceinline__ void stg16_stream(void* p, uint4 v) {
    __stcs(reinterpret_cast<uint4*>(p), v);
}

}  // namespace credit

namespace credit {

}  // namespace credit
