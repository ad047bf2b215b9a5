// pearson.cu -- the Pearson correlation workload: two operands per row.
//
// CREDIT summary page (arXiv 2609.01864v1), "B. Workload-by-Workload
// Scaling" names a Pearson reduction-reuse workload.  Per row of two
// matrices x and u (same shape) the statistics are the means, the biased
// variances and the covariance; h then writes every column's standardized
// co-deviation
//     y_j = (x_j - mx)(u_j - mu) / (sqrt(vx + eps) sqrt(vu + eps)),
// whose row mean is the correlation r, written once per row.
//
// Clustered kernel: the protocol of cluster.cu ("C. Cluster Reduction and
// Reuse Protocol") with two staged slices per CTA -- x at the start of the
// dynamic shared memory, u one pitch further -- so a row is read from HBM
// once and written once (2R + 1W against the re-read baseline's 4R + 1W).
// The CTA partial is (n, mean_x, mean_u) and (Mxx, Muu, Cxu): two 16-byte
// slots per CTA, exchanged with remote stores + cluster barrier or with
// st.async deposits on the receiver's mbarrier.  Co-moments merge in the
// parallel-axis form of Chan et al.:
//     C = sum_q [C_q + n_q (mx_q - mx)(mu_q - mu)],  mx = sum_q n_q mx_q / n.
//
// Two-pass kernels: per (row, chunk) exact two-pass partials into a global
// workspace, then a fold in chunk order and a re-read of both operands.
#include "common.cuh"
#include "internal.h"
#include "rowops.cuh"

namespace credit {

// Thread co-moment sums around shifts K (the thread's first x and u):
// n, sx = sum (x - Kx), su, sxx, suu, sxu.
template <typename T>
struct CoStats {
    F2 nKx = {0.f, 0.f}, nKu = {0.f, 0.f};
    F2 sx = {0.f, 0.f}, su = {0.f, 0.f}, sxx = {0.f, 0.f}, suu = {0.f, 0.f}, sxu = {0.f, 0.f};
    float n = 0.f;
    __device__ __forceinline__ void add(uint4 xr, uint4 ur) {
        constexpr int NP = Pairs<T>::kN;
        F2 px[NP], pu[NP];
        Pairs<T>::unpack(xr, px);
        Pairs<T>::unpack(ur, pu);
        if (n == 0.f) { nKx = f2(-px[0].x); nKu = f2(-pu[0].x); }
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            const F2 dx = add2(px[i], nKx), du = add2(pu[i], nKu);
            sx = add2(sx, dx);
            su = add2(su, du);
            sxx = fma2(dx, dx, sxx);
            suu = fma2(du, du, suu);
            sxu = fma2(dx, du, sxu);
        }
        n += (float)(2 * NP);
    }
    __device__ __forceinline__ void add1(float x, float u) {
        if (n == 0.f) { nKx = f2(-x); nKu = f2(-u); }
        const float dx = x + nKx.x, du = u + nKu.x;
        sx.x += dx;
        su.x += du;
        sxx.x = fmaf(dx, dx, sxx.x);
        suu.x = fmaf(du, du, suu.x);
        sxu.x = fmaf(dx, du, sxu.x);
        n += 1.f;
    }
};

// Partial of a set of elements: count, means, co-moment sums.
struct CoPart {
    float n, mx, mu, mxx, muu, cxu;
};

// Merge of `cnt` partials in order (parallel-axis form, no per-step division).
template <typename Get>
__device__ __forceinline__ CoPart co_merge(int cnt, Get get) {
    float n = 0.f, nx = 0.f, nu = 0.f;
    for (int q = 0; q < cnt; ++q) {
        const CoPart p = get(q);
        n += p.n;
        nx = fmaf(p.n, p.mx, nx);
        nu = fmaf(p.n, p.mu, nu);
    }
    CoPart o;
    o.n = n;
    o.mx = n > 0.f ? nx / n : 0.f;
    o.mu = n > 0.f ? nu / n : 0.f;
    o.mxx = o.muu = o.cxu = 0.f;
    for (int q = 0; q < cnt; ++q) {
        const CoPart p = get(q);
        const float dx = p.mx - o.mx, du = p.mu - o.mu;
        o.mxx += fmaf(p.n * dx, dx, p.mxx);
        o.muu += fmaf(p.n * du, du, p.muu);
        o.cxu += fmaf(p.n * dx, du, p.cxu);
    }
    return o;
}

// The CTA partial from the threads' sums: two block reductions, (n, n mx_t,
// n mu_t) and then the three co-moments about the CTA means.
template <typename T>
__device__ __forceinline__ CoPart co_cta_partial(const CoStats<T>& st, float* redA, float* redB,
                                                 int nwarps, int nthreads) {
    const float n = st.n;
    const float sx = st.sx.x + st.sx.y, su = st.su.x + st.su.y;
    const float mxt = n > 0.f ? sx / n - st.nKx.x : 0.f;
    const float mut = n > 0.f ? su / n - st.nKu.x : 0.f;
    const float mxxt = n > 0.f ? fmaxf(st.sxx.x + st.sxx.y - sx * (sx / n), 0.f) : 0.f;
    const float muut = n > 0.f ? fmaxf(st.suu.x + st.suu.y - su * (su / n), 0.f) : 0.f;
    const float cxut = n > 0.f ? st.sxu.x + st.sxu.y - sx * (su / n) : 0.f;
    float a[3] = {n, n * mxt, n * mut};
    block_reduce_n<3, false>(a, redA, nwarps, nthreads);
    CoPart o;
    o.n = a[0];
    o.mx = a[0] > 0.f ? a[1] / a[0] : 0.f;
    o.mu = a[0] > 0.f ? a[2] / a[0] : 0.f;
    const float dx = mxt - o.mx, du = mut - o.mu;
    float q[3] = {fmaf(n * dx, dx, mxxt), fmaf(n * du, du, muut), fmaf(n * dx, du, cxut)};
    block_reduce_n<3, false>(q, redB, nwarps, nthreads);
    o.mxx = q[0];
    o.muu = q[1];
    o.cxu = q[2];
    return o;
}

// h and r from the row statistics.
struct CoOut {
    float nmx, nmu, inv, r;
    __device__ __forceinline__ CoOut(const CoPart& s, int64_t N, float eps) {
        const float vx = fmaxf(s.mxx / (float)N, 0.f), vu = fmaxf(s.muu / (float)N, 0.f);
        inv = (1.f / sqrtf(vx + eps)) * (1.f / sqrtf(vu + eps));
        nmx = -s.mx;
        nmu = -s.mu;
        r = (s.cxu / (float)N) * inv;
    }
    __device__ __forceinline__ F2 operator()(F2 x, F2 u) const {
        return mul2(mul2(add2(x, f2(nmx)), add2(u, f2(nmu))), f2(inv));
    }
    __device__ __forceinline__ float one(float x, float u) const {
        return ((x + nmx) * (u + nmu)) * inv;
    }
};

template <typename T, bool BULK>
__global__ void __launch_bounds__(kClusterMaxThreads, 3)
cluster_pearson(const ClusterArgs a) {
    using E = Elem<T>;
    constexpr int VEC = E::kVec;
    extern __shared__ __align__(128) unsigned char stage[];
    __shared__ __align__(16) float slots[kMaxCluster * 2 * kSlotStride];
    __shared__ __align__(16) float red[2][kMaxWarps * 3];
    __shared__ __align__(8) uint64_t mbar[kMaxChunks];
    __shared__ __align__(8) uint64_t recv_bar;

    const uint32_t P = cluster_nctarank();
    const uint32_t rank = cluster_ctarank();
    const bool async_x = a.exchange == 1 && P > 1;
    const int64_t row = blockIdx.x / P;
    const int64_t start = (int64_t)rank * a.slice;
    const int n_slice = (int)max((int64_t)0, min(a.cols - start, a.slice));
    // checked build: both staged operands and their chunk mbarriers must fit
    const int n = layout_fits((uint64_t)a.pitch + (uint64_t)n_slice * sizeof(T),
                              BULK ? 2 * (int64_t)((n_slice + a.chunk_elems - 1) / a.chunk_elems) : 0,
                              kMaxChunks, a.err)
                      ? n_slice : 0;
    const T* xs = static_cast<const T*>(a.x) + row * a.cols + start;
    const T* us = static_cast<const T*>(a.p0) + row * a.cols + start;
    unsigned char* ustage = stage + a.pitch;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31, nwarps = nt >> 5;
    const int nvec = n / VEC;

    if (async_x && tid == 0) {
        // two arrivals (this one, registering the peers' two 16-byte deposits
        // each before any peer passes the entry barrier, and the local store
        // of this CTA's own partial) plus those bytes
        const uint32_t rb = smem_u32(&recv_bar);
        mbar_init(rb, 2);
        mbar_arrive_expect_tx(rb, (P - 1) * 2u * 16u);
        fence_mbar_init();
    }
    if (P > 1) cluster_arrive_relaxed();

    // ---------------------------------------------------------- stage x, u
    int cpr = 1, vpc = nvec;
    if constexpr (BULK) {
        cpr = (n + a.chunk_elems - 1) / a.chunk_elems;
        vpc = a.chunk_elems / VEC;
        if (tid == 0) {
            for (int c = 0; c < 2 * cpr; ++c) mbar_init(smem_u32(&mbar[c]), 1);
            fence_mbar_init();
            fence_proxy_async_smem();
            const uint64_t pol = l2_policy_evict_first();
            for (int c = 0; c < cpr; ++c) {
                const int e0 = c * a.chunk_elems;
                const uint32_t bytes = (uint32_t)(min(a.chunk_elems, n - e0) * (int)sizeof(T));
                const uint32_t off = (uint32_t)(e0 * (int)sizeof(T));
                const uint32_t bx = smem_u32(&mbar[2 * c]), bu = smem_u32(&mbar[2 * c + 1]);
                mbar_arrive_expect_tx(bx, bytes);
                bulk_g2s(smem_u32(stage) + off, xs + e0, bytes, bx, pol);
                mbar_arrive_expect_tx(bu, bytes);
                bulk_g2s(smem_u32(ustage) + off, us + e0, bytes, bu, pol);
            }
        }
        __syncthreads();
    } else {
        T* sx = reinterpret_cast<T*>(stage);
        T* su = reinterpret_cast<T*>(ustage);
        for (int i = tid; i < n; i += nt) { sx[i] = xs[i]; su[i] = us[i]; }
        __syncthreads();
    }
    auto xat = [&](int i) { return E::to_f(reinterpret_cast<const T*>(stage)[i]); };
    auto uat = [&](int i) { return E::to_f(reinterpret_cast<const T*>(ustage)[i]); };

    // ------------------------------------------------------ local partial
    CoStats<T> st;
    for (int c = 0; c < cpr; ++c) {
        if constexpr (BULK) {
            mbar_wait_bounded(smem_u32(&mbar[2 * c]), 0, a.err);
            mbar_wait_bounded(smem_u32(&mbar[2 * c + 1]), 0, a.err);
        }
        const int v0 = c * vpc, v1 = min(nvec, v0 + vpc);
        for_tiles<4>(v1 - v0, warp, nwarps, lane, [&](int v) {
            const size_t o = (size_t)(v0 + v) * 16;
            st.add(lds16(stage + o), lds16(ustage + o));
        });
    }
    if constexpr (!BULK) {
        for (int i = nvec * VEC + tid; i < n; i += nt) st.add1(xat(i), uat(i));
    }
    const CoPart part = co_cta_partial<T>(st, red[0], red[1], nwarps, nt);

    // ------------------------------------------- exchange and combine
    CoPart tot = part;
    if (P > 1) {
        cluster_wait_acquire();  // every peer has started
        const float v0[4] = {part.n, part.mx, part.mu, 0.f};
        const float v1[4] = {part.mxx, part.muu, part.cxu, 0.f};
        if (async_x) {
            if (tid == (int)rank) {
                float* d = &slots[rank * 2 * kSlotStride];
                for (int k = 0; k < 4; ++k) { d[k] = v0[k]; d[kSlotStride + k] = v1[k]; }
                mbar_arrive(smem_u32(&recv_bar));
            } else if (tid < (int)P) {
                const uint32_t rbar = mapa_shared(smem_u32(&recv_bar), (uint32_t)tid);
                const uint32_t dst = mapa_shared(smem_u32(&slots[rank * 2 * kSlotStride]), (uint32_t)tid);
                st_async_v4f32(dst, v0[0], v0[1], v0[2], v0[3], rbar);
                st_async_v4f32(dst + 16u, v1[0], v1[1], v1[2], v1[3], rbar);
            }
            mbar_wait_bounded(smem_u32(&recv_bar), 0, a.err);
            cluster_arrive_relaxed();
        } else {
            if (tid < (int)P) {
                const uint32_t dst = mapa_shared(smem_u32(&slots[rank * 2 * kSlotStride]), (uint32_t)tid);
                st_cluster_v4f32(dst, v0[0], v0[1], v0[2], v0[3]);
                st_cluster_v4f32(dst + 16u, v1[0], v1[1], v1[2], v1[3]);
            }
            cluster_arrive_release();
            cluster_wait_acquire();
        }
        tot = co_merge((int)P, [&](int q) {
            const float* s = &slots[q * 2 * kSlotStride];
            return CoPart{s[0], s[1], s[2], s[kSlotStride], s[kSlotStride + 1], s[kSlotStride + 2]};
        });
    }

    if (tid == 0) {
        const float v[6] = {tot.n, tot.mx, tot.mu, tot.mxx, tot.muu, tot.cxu};
        debug_row_stats(a.dbg_stats, row, rank, P, v, 6);
    }
    // ---------------------------------------------------------- output
    const CoOut h(tot, a.cols, a.eps);
    if (rank == 0 && tid == 0) a.aux[row] = h.r;
    T* yrow = static_cast<T*>(a.y) + row * a.cols + start;
    if constexpr (BULK) {
        constexpr int NP = Pairs<T>::kN;
        for_tiles<4>(nvec, warp, nwarps, lane, [&](int v) {
            F2 px[NP], pu[NP];
            Pairs<T>::unpack(lds16(stage + (size_t)v * 16), px);
            Pairs<T>::unpack(lds16(ustage + (size_t)v * 16), pu);
#pragma unroll
            for (int i = 0; i < NP; ++i) px[i] = h(px[i], pu[i]);
            stg16_stream(reinterpret_cast<uint4*>(yrow) + v, Pairs<T>::pack(px));
        });
    } else {
        for (int i = tid; i < n; i += nt) yrow[i] = E::from_f(h.one(xat(i), uat(i)));
    }
    // st.async exchange: keep every CTA alive until all deposits have landed
    if (async_x) cluster_wait_acquire();
}

// ------------------------------------------------------------ two-pass
template <typename T, bool VEC_PATH>
__device__ __forceinline__ void load_chunk(const T* p, int64_t n, float* f, bool* ok) {
    constexpr int kV = Elem<T>::kVec;
#pragma unroll
    for (int k = 0; k < kTwoPassVpt; ++k) {
        const int64_t e0 = ((int64_t)k * blockDim.x + threadIdx.x) * kV;
        if constexpr (VEC_PATH) {
            if (e0 < n) {
                Elem<T>::unpack(*reinterpret_cast<const uint4*>(p + e0), &f[k * kV]);
#pragma unroll
                for (int i = 0; i < kV; ++i) ok[k * kV + i] = true;
            } else {
#pragma unroll
                for (int i = 0; i < kV; ++i) { ok[k * kV + i] = false; f[k * kV + i] = 0.f; }
            }
        } else {
#pragma unroll
            for (int i = 0; i < kV; ++i) {
                const bool in = e0 + i < n;
                ok[k * kV + i] = in;
                f[k * kV + i] = in ? Elem<T>::to_f(p[e0 + i]) : 0.f;
            }
        }
    }
}

// exact two-pass partial of one (row, chunk): means, then co-moment sums
template <typename T, bool VEC_PATH>
__global__ void __launch_bounds__(kMaxThreads)
pearson_stats(const TwoPassArgs a) {
    __shared__ float red[5][kMaxWarps];
    constexpr int N = kTwoPassVpt * Elem<T>::kVec;
    const int64_t row = blockIdx.y;
    const int c = blockIdx.x;
    const int64_t j0 = (int64_t)c * a.chunk;
    const int64_t n = min((int64_t)a.chunk, a.cols - j0);
    float fx[N], fu[N];
    bool ok[N];
    load_chunk<T, VEC_PATH>(static_cast<const T*>(a.x) + row * a.cols + j0, n, fx, ok);
    load_chunk<T, VEC_PATH>(static_cast<const T*>(a.p0) + row * a.cols + j0, n, fu, ok);
    float sx = 0.f, su = 0.f;
#pragma unroll
    for (int e = 0; e < N; ++e) { sx += fx[e]; su += fu[e]; }  // masked entries are 0
    sx = block_allreduce(sx, red[0], SumOp{}, 0.f);
    su = block_allreduce(su, red[1], SumOp{}, 0.f);
    const float mx = sx / (float)n, mu = su / (float)n;
    float sxx = 0.f, suu = 0.f, sxu = 0.f;
#pragma unroll
    for (int e = 0; e < N; ++e) {
        if (ok[e]) {
            const float dx = fx[e] - mx, du = fu[e] - mu;
            sxx = fmaf(dx, dx, sxx);
            suu = fmaf(du, du, suu);
            sxu = fmaf(dx, du, sxu);
        }
    }
    sxx = block_allreduce(sxx, red[2], SumOp{}, 0.f);
    suu = block_allreduce(suu, red[3], SumOp{}, 0.f);
    sxu = block_allreduce(sxu, red[4], SumOp{}, 0.f);
    if (threadIdx.x == 0) {
        float4* w = reinterpret_cast<float4*>(a.ws) + 2 * (row * a.nch + c);
        w[0] = make_float4((float)n, mx, mu, 0.f);
        w[1] = make_float4(sxx, suu, sxu, 0.f);
    }
}

template <typename T, bool VEC_PATH>
__global__ void __launch_bounds__(kMaxThreads)
pearson_apply(const TwoPassArgs a) {
    using E = Elem<T>;
    constexpr int kV = E::kVec, N = kTwoPassVpt * kV;
    const int64_t row = blockIdx.y;
    const int c = blockIdx.x;
    const int64_t j0 = (int64_t)c * a.chunk;
    const int64_t n = min((int64_t)a.chunk, a.cols - j0);
    const float4* w = reinterpret_cast<const float4*>(a.ws) + 2 * row * a.nch;
    const CoPart tot = co_merge(a.nch, [&](int q) {
        const float4 p = w[2 * q], m = w[2 * q + 1];
        return CoPart{p.x, p.y, p.z, m.x, m.y, m.z};
    });
    const CoOut h(tot, a.cols, a.eps);
    if (c == 0 && threadIdx.x == 0) a.aux[row] = h.r;
    // the re-read of both operands
    float fx[N], fu[N];
    bool ok[N];
    load_chunk<T, VEC_PATH>(static_cast<const T*>(a.x) + row * a.cols + j0, n, fx, ok);
    load_chunk<T, VEC_PATH>(static_cast<const T*>(a.p0) + row * a.cols + j0, n, fu, ok);
    T* ys = static_cast<T*>(a.y) + row * a.cols + j0;
#pragma unroll
    for (int k = 0; k < kTwoPassVpt; ++k) {
        const int64_t e0 = ((int64_t)k * blockDim.x + threadIdx.x) * kV;
        if (e0 >= n) break;
        float* f = &fx[k * kV];
#pragma unroll
        for (int i = 0; i < kV; ++i) f[i] = h.one(f[i], fu[k * kV + i]);
        if constexpr (VEC_PATH) {
            st_global_cs_v4(ys + e0, E::pack(f));
        } else {
#pragma unroll
            for (int i = 0; i < kV; ++i) if (e0 + i < n) ys[e0 + i] = E::from_f(f[i]);
        }
    }
}

// ------------------------------------------------------------ dispatch
const void* pearson_cluster_kernel(int dtype, bool vec) {
    if (dtype == 0) return vec ? (const void*)cluster_pearson<float, true>
                               : (const void*)cluster_pearson<float, false>;
    return vec ? (const void*)cluster_pearson<bf16, true> : (const void*)cluster_pearson<bf16, false>;
}

const void* pearson_stats_kernel(int dtype, bool vec) {
    if (dtype == 0) return vec ? (const void*)pearson_stats<float, true>
                               : (const void*)pearson_stats<float, false>;
    return vec ? (const void*)pearson_stats<bf16, true> : (const void*)pearson_stats<bf16, false>;
}

const void* pearson_apply_kernel(int dtype, bool vec) {
    if (dtype == 0) return vec ? (const void*)pearson_apply<float, true>
                               : (const void*)pearson_apply<float, false>;
    return vec ? (const void*)pearson_apply<bf16, true> : (const void*)pearson_apply<bf16, false>;
}

}  // namespace credit
