// two_pass.cu -- the non-clustered baseline: partial statistics per
// (row, chunk) into a global workspace, then a second kernel that folds the
// row's partials, RE-READS the chunk from global memory and writes the
// output.  This is the "global re-read" arm of the non-DSMEM CUDA baseline
// on the CREDIT summary page (arXiv 2609.01864v1, "A. Experimental Setup and
// Baselines"); it moves 2 reads + 1 write per element, and the difference to
// the clustered kernel's 1 read + 1 write is exactly the re-read traffic the
// transformation removes ("B. Reduction-Reuse Transformation", traffic model).
//
// Each block holds its chunk in registers (kTwoPassVpt 16-byte vectors per
// thread), so its partial is an exact two-pass over the chunk: max then
// sum-exp (softmax), mean then squared deviations (LayerNorm), or a sum of
// squares (RMSNorm).  Partials are folded in chunk order, so every block of a
// row sees identical statistics.
#include "common.cuh"
#include "internal.h"

namespace credit {

template <typename T, bool VEC_PATH>
struct ChunkRegs {
    static constexpr int kVec = Elem<T>::kVec;
    static constexpr int kN = kTwoPassVpt * kVec;  // elements per thread
    float f[kN];
    bool ok[kTwoPassVpt * kVec];

    // element e of this thread's share: vector slot k, lane i -> column
    // j0 + (k * nt + tid) * VEC + i (coalesced 16-byte accesses).
    __device__ void load(const T* xs, int64_t n, int tid, int nt) {
#pragma unroll
        for (int k = 0; k < kTwoPassVpt; ++k) {
            const int64_t e0 = ((int64_t)k * nt + tid) * kVec;
            if constexpr (VEC_PATH) {
                if (e0 < n) {
                    Elem<T>::unpack(*reinterpret_cast<const uint4*>(xs + e0), &f[k * kVec]);
#pragma unroll
                    for (int i = 0; i < kVec; ++i) ok[k * kVec + i] = true;
                } else {
#pragma unroll
                    for (int i = 0; i < kVec; ++i) { ok[k * kVec + i] = false; f[k * kVec + i] = 0.f; }
                }
            } else {
#pragma unroll
                for (int i = 0; i < kVec; ++i) {
                    const bool in = e0 + i < n;
                    ok[k * kVec + i] = in;
                    f[k * kVec + i] = in ? Elem<T>::to_f(xs[e0 + i]) : 0.f;
                }
            }
        }
    }
};

template <int OP, typename T, typename PT, bool VEC_PATH>
__global__ void __launch_bounds__(kMaxThreads)
two_pass_stats(const TwoPassArgs a) {
    __shared__ float red[2][kMaxWarps];
    const int64_t row = blockIdx.y;
    const int c = blockIdx.x;
    const int64_t j0 = (int64_t)c * a.chunk;
    const int64_t n = min((int64_t)a.chunk, a.cols - j0);
    const T* xs = static_cast<const T*>(a.x) + row * a.cols + j0;
    ChunkRegs<T, VEC_PATH> r;
    r.load(xs, n, threadIdx.x, blockDim.x);
    constexpr int N = ChunkRegs<T, VEC_PATH>::kN;

    float p0 = 0.f, p1 = 0.f, p2 = 0.f;
    if constexpr (OP == kQuant) {
        float m = 0.f;
#pragma unroll
        for (int e = 0; e < N; ++e) m = fmaxf(m, fabsf(r.f[e]));  // masked entries are 0
        p0 = block_allreduce(m, red[0], MaxOp{}, 0.f);
    } else if constexpr (OP == kWStd) {
        // weights of this thread's elements, then an exact two-pass over the chunk
        float w[N];
        const PT* wp = static_cast<const PT*>(a.p0) + j0;
        constexpr int kV = Elem<T>::kVec;
#pragma unroll
        for (int k = 0; k < kTwoPassVpt; ++k) {
            const int64_t e0 = ((int64_t)k * blockDim.x + threadIdx.x) * kV;
#pragma unroll
            for (int i = 0; i < kV; ++i)
                w[k * kV + i] = (e0 + i < n) ? load_param1<PT>(wp, e0 + i) : 0.f;
        }
        float sw = 0.f, swx = 0.f;
#pragma unroll
        for (int e = 0; e < N; ++e) { sw += w[e]; swx = fmaf(w[e], r.f[e], swx); }
        sw = block_allreduce(sw, red[0], SumOp{}, 0.f);
        swx = block_allreduce(swx, red[1], SumOp{}, 0.f);
        const float mu = sw > 0.f ? swx / sw : 0.f;
        float m2 = 0.f;
#pragma unroll
        for (int e = 0; e < N; ++e) { const float d = r.f[e] - mu; m2 = fmaf(w[e] * d, d, m2); }
        __syncthreads();  // red[0] is reused below
        m2 = block_allreduce(m2, red[0], SumOp{}, 0.f);
        p0 = sw; p1 = mu; p2 = m2;
    } else if constexpr (OP == kSoftmax) {
        float m = -INFINITY;
#pragma unroll
        for (int e = 0; e < N; ++e) if (r.ok[e]) m = fmaxf(m, r.f[e]);
        m = block_allreduce(m, red[0], MaxOp{}, -INFINITY);
        const float ml = m * kLog2e;
        float s = 0.f;
#pragma unroll
        for (int e = 0; e < N; ++e) if (r.ok[e]) s += exp_shift<T>(r.f[e], m, ml);
        s = block_allreduce(s, red[1], SumOp{}, 0.f);
        p0 = m; p1 = s;
    } else if constexpr (OP == kLayerNorm) {
        float s = 0.f;
#pragma unroll
        for (int e = 0; e < N; ++e) s += r.f[e];  // masked entries are 0
        s = block_allreduce(s, red[0], SumOp{}, 0.f);
        const float mu = s / (float)n;
        float m2 = 0.f;
#pragma unroll
        for (int e = 0; e < N; ++e) if (r.ok[e]) { const float d = r.f[e] - mu; m2 = fmaf(d, d, m2); }
        m2 = block_allreduce(m2, red[1], SumOp{}, 0.f);
        p0 = (float)n; p1 = mu; p2 = m2;
    } else {
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < N; ++e) ss = fmaf(r.f[e], r.f[e], ss);
        ss = block_allreduce(ss, red[0], SumOp{}, 0.f);
        p0 = ss;
    }
    if (threadIdx.x == 0) {
        float4* w = reinterpret_cast<float4*>(a.ws) + row * a.nch + c;
        *w = make_float4(p0, p1, p2, 0.f);
    }
}

template <int OP, typename T, typename PT, bool VEC_PATH>
__global__ void __launch_bounds__(kMaxThreads)
two_pass_apply(const TwoPassArgs a) {
    using E = Elem<T>;
    constexpr int VEC = E::kVec;
    const int64_t row = blockIdx.y;
    const int c = blockIdx.x;
    const int64_t j0 = (int64_t)c * a.chunk;
    const int64_t n = min((int64_t)a.chunk, a.cols - j0);
    const float4* w = reinterpret_cast<const float4*>(a.ws) + row * a.nch;

    // fold the row's partials in chunk order (identical in every block)
    float c0, c1 = 0.f;
    if constexpr (OP == kQuant) {
        float m = 0.f;
        for (int q = 0; q < a.nch; ++q) m = fmaxf(m, w[q].x);
        c0 = m / 127.f;  // the row scale (IEEE division)
        if (c == 0 && threadIdx.x == 0) a.aux[row] = c0;
    } else if constexpr (OP == kWStd) {
        float W = 0.f, wm = 0.f;
        for (int q = 0; q < a.nch; ++q) { const float4 v = w[q]; W += v.x; wm = fmaf(v.x, v.y, wm); }
        const float mean = W > 0.f ? wm / W : 0.f;
        float m2 = 0.f;
        for (int q = 0; q < a.nch; ++q) {
            const float4 v = w[q];
            const float d = v.y - mean;
            m2 += fmaf(v.x * d, d, v.z);
        }
        const float rr = 1.f / sqrtf(fmaxf(W > 0.f ? m2 / W : 0.f, 0.f) + a.eps);
        c0 = rr;
        c1 = -mean * rr;
    } else if constexpr (OP == kSoftmax) {
        float m = -INFINITY;
        for (int q = 0; q < a.nch; ++q) m = fmaxf(m, w[q].x);
        float s = 0.f;
        for (int q = 0; q < a.nch; ++q) { const float4 v = w[q]; s += rescale(v.y, v.x, m); }
        if constexpr (sizeof(T) == 4) { c0 = m; c1 = 1.f / s; }
        else { c0 = m * kLog2e; c1 = 1.f / s; }
    } else if constexpr (OP == kLayerNorm) {
        NormPart acc{0.f, 0.f, 0.f};
        for (int q = 0; q < a.nch; ++q) { const float4 v = w[q]; acc = chan_merge(acc, NormPart{v.x, v.y, v.z}); }
        c0 = acc.mu;
        c1 = 1.f / sqrtf(fmaxf(acc.m2 / (float)a.cols, 0.f) + a.eps);
    } else {
        float ss = 0.f;
        for (int q = 0; q < a.nch; ++q) ss += w[q].x;
        c0 = 1.f / sqrtf(ss / (float)a.cols + a.eps);
    }

    // the re-read
    const T* xs = static_cast<const T*>(a.x) + row * a.cols + j0;
    T* ys = static_cast<T*>(a.y) + row * a.cols + j0;
    ChunkRegs<T, VEC_PATH> r;
    r.load(xs, n, threadIdx.x, blockDim.x);
    if constexpr (OP == kQuant) {
        int8_t* qs = static_cast<int8_t*>(a.y) + row * a.cols + j0;
        const float inv = quant_inv(c0);
        constexpr int kV = Elem<T>::kVec;
#pragma unroll
        for (int k = 0; k < kTwoPassVpt; ++k) {
            const int64_t e0 = ((int64_t)k * blockDim.x + threadIdx.x) * kV;
            if constexpr (VEC_PATH) {
                // whole vectors: kV codes packed into 4 or 8 bytes
                if (e0 < n) {
                    float xf[kV];
#pragma unroll
                    for (int i = 0; i < kV; ++i) xf[i] = r.f[k * kV + i];
                    uint32_t w[kV / 4];
                    quant_codes<kV>(xf, c0, inv, w);
                    if constexpr (kV == 4) __stcs(reinterpret_cast<unsigned int*>(qs + e0), w[0]);
                    else __stcs(reinterpret_cast<uint2*>(qs + e0), make_uint2(w[0], w[1]));
                }
            } else {
#pragma unroll
                for (int i = 0; i < kV; ++i)
                    if (e0 + i < n) qs[e0 + i] = (int8_t)quant_code(r.f[k * kV + i], c0, inv);
            }
        }
        return;
    }
    const PT* g = static_cast<const PT*>(a.p0);
    const PT* b = static_cast<const PT*>(a.p1);
#pragma unroll
    for (int k = 0; k < kTwoPassVpt; ++k) {
        const int64_t e0 = ((int64_t)k * blockDim.x + threadIdx.x) * VEC;
        if (e0 >= n) break;
        float* f = &r.f[k * VEC];
        float gv[VEC], bv[VEC];
#pragma unroll
        for (int i = 0; i < VEC; ++i) { gv[i] = 1.f; bv[i] = 0.f; }
        if constexpr (OP == kLayerNorm || OP == kRMSNorm) {
            if constexpr (VEC_PATH) {
                if (g) load_params<PT, VEC>(g, j0 + e0, gv);
                if (b) load_params<PT, VEC>(b, j0 + e0, bv);
            } else {
#pragma unroll
                for (int i = 0; i < VEC; ++i) {
                    if (e0 + i < n) {
                        if (g) gv[i] = load_param1<PT>(g, j0 + e0 + i);
                        if (b) bv[i] = load_param1<PT>(b, j0 + e0 + i);
                    }
                }
            }
        }
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            if constexpr (OP == kWStd) {
                f[i] = fmaf(f[i], c0, c1);
            } else if constexpr (OP == kSoftmax) {
                if constexpr (sizeof(T) == 4) f[i] = expf(f[i] - c0) * c1;
                else f[i] = fast_ex2(fmaf(f[i], kLog2e, -c0)) * c1;
            } else if constexpr (OP == kLayerNorm) {
                f[i] = fmaf((f[i] - c0) * c1, gv[i], bv[i]);
            } else {
                f[i] = (f[i] * c0) * gv[i];
            }
        }
        if constexpr (VEC_PATH) {
            st_global_cs_v4(ys + e0, E::pack(f));
        } else {
#pragma unroll
            for (int i = 0; i < VEC; ++i) if (e0 + i < n) ys[e0 + i] = E::from_f(f[i]);
        }
    }
}

// ----------------------------------------------------------- dispatch
template <int OP, typename T, typename PT>
static const void* stats_pick(bool vec) {
    return vec ? (const void*)two_pass_stats<OP, T, PT, true>
               : (const void*)two_pass_stats<OP, T, PT, false>;
}

template <int OP, typename T>
static const void* stats_param(int pdtype, bool vec) {
    return pdtype == 0 ? stats_pick<OP, T, float>(vec) : stats_pick<OP, T, bf16>(vec);
}

const void* two_pass_stats_kernel(KernelKey k) {
    switch (k.op) {
        case kSoftmax: return k.dtype == 0 ? stats_pick<kSoftmax, float, float>(k.vec) : stats_pick<kSoftmax, bf16, float>(k.vec);
        case kLayerNorm: return k.dtype == 0 ? stats_pick<kLayerNorm, float, float>(k.vec) : stats_pick<kLayerNorm, bf16, float>(k.vec);
        case kRMSNorm: return k.dtype == 0 ? stats_pick<kRMSNorm, float, float>(k.vec) : stats_pick<kRMSNorm, bf16, float>(k.vec);
        case kQuant: return k.dtype == 0 ? stats_pick<kQuant, float, float>(k.vec) : stats_pick<kQuant, bf16, float>(k.vec);
        case kWStd: return k.dtype == 0 ? stats_param<kWStd, float>(k.pdtype, k.vec) : stats_param<kWStd, bf16>(k.pdtype, k.vec);
        case kPearson: return pearson_stats_kernel(k.dtype, k.vec);
    }
    return nullptr;
}

template <int OP, typename T, typename PT>
static const void* apply_pick(bool vec) {
    return vec ? (const void*)two_pass_apply<OP, T, PT, true> : (const void*)two_pass_apply<OP, T, PT, false>;
}

template <int OP>
static const void* apply_dtype(int dtype, int pdtype, bool vec) {
    if (dtype == 0) return pdtype == 0 ? apply_pick<OP, float, float>(vec) : apply_pick<OP, float, bf16>(vec);
    return pdtype == 0 ? apply_pick<OP, bf16, float>(vec) : apply_pick<OP, bf16, bf16>(vec);
}

const void* two_pass_apply_kernel(KernelKey k) {
    switch (k.op) {
        case kSoftmax: return k.dtype == 0 ? apply_pick<kSoftmax, float, float>(k.vec)
                                           : apply_pick<kSoftmax, bf16, float>(k.vec);
        case kLayerNorm: return apply_dtype<kLayerNorm>(k.dtype, k.pdtype, k.vec);
        case kRMSNorm: return apply_dtype<kRMSNorm>(k.dtype, k.pdtype, k.vec);
        case kQuant: return k.dtype == 0 ? apply_pick<kQuant, float, float>(k.vec)
                                         : apply_pick<kQuant, bf16, float>(k.vec);
        case kWStd: return apply_dtype<kWStd>(k.dtype, k.pdtype, k.vec);
        case kPearson: return pearson_apply_kernel(k.dtype, k.vec);
    }
    return nullptr;
}

cudaError_t launch_two_pass(KernelKey k, const TwoPassArgs& a, int64_t rows, int threads,
                            cudaStream_t s) {
    const void* fs = two_pass_stats_kernel(k);
    const void* fa = two_pass_apply_kernel(k);
    if (!fs || !fa) return cudaErrorInvalidDeviceFunction;
    const size_t esz = k.dtype == 0 ? 4 : 2;
    const size_t yesz = k.op == kQuant ? 1 : esz;  // int8 codes
    const int64_t max_rows = 65535;  // gridDim.y limit
    for (int64_t r0 = 0; r0 < rows; r0 += max_rows) {
        const int64_t nr = rows - r0 < max_rows ? rows - r0 : max_rows;
        TwoPassArgs b = a;
        b.x = static_cast<const char*>(a.x) + r0 * a.cols * (int64_t)esz;
        b.y = static_cast<char*>(a.y) + r0 * a.cols * (int64_t)yesz;
        b.ws = a.ws + r0 * a.nch * (k.op == kPearson ? 8 : 4);
        if (a.aux) b.aux = a.aux + r0;
        if (k.op == kPearson) b.p0 = static_cast<const char*>(a.p0) + r0 * a.cols * (int64_t)esz;
        void* args[] = {&b};
        const dim3 grid((unsigned)a.nch, (unsigned)nr, 1);
        cudaError_t e = cudaLaunchKernel(fs, grid, dim3((unsigned)threads), args, 0, s);
        if (e != cudaSuccess) return e;
        e = cudaLaunchKernel(fa, grid, dim3((unsigned)threads), args, 0, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace credit
