// persistent.cu -- the clustered reduce-reuse kernel as a persistent,
// warp-specialised pipeline.
//
// The grid holds only the clusters that can be resident at once; cluster
// `cid` handles rows cid, cid + G, cid + 2G, ...  Every CTA owns the same
// column slice of each of those rows (CREDIT summary page, arXiv
// 2609.01864v1, "B. Reduction-Reuse Transformation": P non-overlapping
// CTA-owned slices).  Per CTA:
//   - one producer warp streams the slice of row after row into a ring of
//     shared-memory slots with non-multicast bulk copies, one "full" mbarrier
//     per slot (transaction bytes) and one "empty" mbarrier per slot (one
//     arrival per consumer warp once the slot's output has been written);
//   - the consumer warps, per row: fold each chunk into per-thread partials
//     as it lands, merge them into the CTA partial, push it into slot `rank`
//     of every peer (mapa + st.shared::cluster), pass the cluster barrier,
//     combine the P slots in rank order, apply h to the whole staged slice
//     and release the row's slots back to the producer ("C. Cluster
//     Reduction and Reuse Protocol").
// The ring holds at least one whole slice, so the row is read from HBM once;
// when it holds two or more, the next row's copies are in flight while this
// row reduces, exchanges and writes.
// Slot arrays are double-buffered by row parity: the cluster barrier of row k
// orders every read of row k-1's slots before any push of row k+1, which is
// the job of the page's second barrier.  A relaxed arrive at entry, waited on
// before the first push, guarantees every peer is running.
// Every wait on an mbarrier is bounded (a second); the producer warp takes
// part in each cluster barrier phase one row ahead of the consumers.
#include "common.cuh"
#include "internal.h"
#include "rowops.cuh"

namespace credit {

template <int OP, typename T, typename PT>
__global__ void __launch_bounds__(kPersistMaxThreads, 1)
cluster_persistent(const PersistArgs a) {
    using E = Elem<T>;
    constexpr int VEC = E::kVec;
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(16) float slots[2][kMaxCluster * kSlotStride];
    __shared__ __align__(16) float red[2][2][(kPersistMaxThreads / 32) * 2];  // [row parity][stage]
    __shared__ __align__(8) uint64_t full_bar[kPersistMaxSlots];
    __shared__ __align__(8) uint64_t empty_bar[kPersistMaxSlots];
    __shared__ __align__(8) uint64_t recv_bar[2];  // st.async exchange, by row parity

    const uint32_t P = cluster_nctarank();
    const uint32_t rank = cluster_ctarank();
    const int64_t cid = blockIdx.x / P;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int ncw = (int)(blockDim.x >> 5) - 1;  // consumer warps; the last warp produces
    const int nct = ncw * 32;
    const int64_t start = (int64_t)rank * a.slice;
    const int cpr_full = (a.slice + a.chunk - 1) / a.chunk;  // slots per row slot
    const int NR = a.nslots / cpr_full;                 // rows the ring holds
    // checked build: the ring's slots and bytes must fit the launch
    const bool fits = layout_fits((uint64_t)a.nslots * a.chunk * sizeof(T), (int64_t)NR * cpr_full,
                                  kPersistMaxSlots, a.err);
    const int n = fits ? (int)max((int64_t)0, min(a.cols - start, (int64_t)a.slice)) : 0;
    const int nvec = n / VEC;
    const int vpc = a.chunk / VEC;                      // vectors per slot
    const int cpr = (n + a.chunk - 1) / a.chunk;        // chunks this CTA stages per row
    const uint32_t ring_s = smem_u32(ring);             // shared-window address for the bulk copies
    const uint32_t slot_bytes = (uint32_t)a.chunk * (uint32_t)sizeof(T);
    const int64_t nrows = cid < a.rows ? (a.rows - 1 - cid) / a.nclusters + 1 : 0;
    const bool clustered = P > 1;
    const bool async_x = clustered && a.exchange == 1;
    const uint32_t xbytes = (P - 1) * 16u;  // the peers' deposits of one row
    // Row k of this CTA lives in row slot k mod NR: slots
    // [rs * cpr_full, rs * cpr_full + cpr), contiguous in shared memory; the
    // slot's use count is k div NR.  Both are tracked incrementally.

    if (tid == 0) {
        for (int s = 0; s < (fits ? NR * cpr_full : 0); ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), (uint32_t)ncw);
        }
        if (async_x) {
            // two arrivals per row: the expected bytes (posted here for rows
            // 0 and 1, after each wait for row k + 2) and the local partial
            for (int b = 0; b < 2; ++b) {
                mbar_init(smem_u32(&recv_bar[b]), 2);
                if (b < nrows) mbar_arrive_expect_tx(smem_u32(&recv_bar[b]), xbytes);
            }
        }
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    __syncthreads();
    if (clustered) cluster_arrive_relaxed();

    // ------------------------------------------------------------ producer
    if (warp == ncw) {
        const uint64_t pol = l2_policy_evict_first();
        int rs = 0;
        uint32_t use = 0;
        for (int64_t k = 0; k < nrows; ++k) {
            if (lane == 0) {
                const T* src = static_cast<const T*>(a.x) + (cid + k * a.nclusters) * a.cols + start;
                for (int c = 0; c < cpr; ++c) {
                    const int slot = rs * cpr_full + c;
                    if (use > 0) mbar_wait_bounded(smem_u32(&empty_bar[slot]), (use - 1) & 1u, a.err);
                    const int e0 = c * a.chunk;
                    const uint32_t bytes = (uint32_t)(min(a.chunk, n - e0) * (int)sizeof(T));
                    const uint32_t fb = smem_u32(&full_bar[slot]);
                    mbar_arrive_expect_tx(fb, bytes);
                    bulk_g2s(ring_s + (uint32_t)slot * slot_bytes, src + e0, bytes, fb, pol);
                }
            }
            if (++rs == NR) { rs = 0; ++use; }
            __syncwarp();
            if (clustered && !async_x) {
                cluster_wait_acquire();   // entry phase (k == 0) or row k-1
                cluster_arrive_relaxed(); // row k
            }
        }
        if (async_x) {
            cluster_wait_acquire();       // the entry phase
            cluster_arrive_relaxed();     // the exit phase
        }
        if (clustered) cluster_wait_acquire();  // last row (or the entry / exit phase)
        return;
    }

    // ----------------------------------------------------------- consumers
    const PT* gp = static_cast<const PT*>(a.p0);
    const PT* bp = static_cast<const PT*>(a.p1);
    int rs = 0;
    uint32_t use = 0;
    for (int64_t k = 0; k < nrows; ++k) {
        const int64_t row = cid + k * a.nclusters;
        unsigned char* base = ring + (size_t)rs * cpr_full * slot_bytes;  // the staged slice

        // a2 + a3: fold each chunk into the thread's statistics as it lands
        Stats<OP, T> stt;
        for (int c = 0; c < cpr; ++c) {
            mbar_wait_bounded(smem_u32(&full_bar[rs * cpr_full + c]), use & 1u, a.err);
            const int v0 = c * vpc;
            stats_tiles(stt, base + (size_t)v0 * 16, min(nvec, v0 + vpc) - v0, warp, ncw, lane);
        }
        auto stash = [&](float mq) { return softmax_stash(base, nvec, warp, ncw, lane, mq); };
        float p0, p1, p2;
        cta_partial<OP, T>(stt, red[k & 1][0], red[k & 1][1], ncw, nct, stash, p0, p1, p2);
        // the fp32 softmax stash wrote the slots: order those generic-proxy
        // writes before the bulk copies that will refill them
        if constexpr (OP == kSoftmax && sizeof(T) == 4) fence_proxy_async_smem();

        // a4 + a5 + a6: replicated push, cluster barrier, local combine
        float st0 = p0, st1 = p1, st2 = p2;
        if (clustered) {
            if (k == 0) cluster_wait_acquire();  // every peer is running
            float* sl = slots[k & 1];
            if (async_x) {
                // thread t deposits into peer t; thread `rank` stores locally
                const uint32_t rb = smem_u32(&recv_bar[k & 1]);
                if (tid == (int)rank) {
                    float* d = &sl[rank * kSlotStride];
                    d[0] = p0; d[1] = p1; d[2] = p2;
                    mbar_arrive(rb);
                } else if (tid < (int)P) {
                    const uint32_t dst = mapa_shared(smem_u32(&sl[rank * kSlotStride]), (uint32_t)tid);
                    st_async_v4f32(dst, p0, p1, p2, 0.f, mapa_shared(rb, (uint32_t)tid));
                }
                mbar_wait_bounded(rb, (uint32_t)(k >> 1) & 1u, a.err);
                // this slot array's next row (k + 2) expects its deposits;
                // no peer can deposit them before this CTA's row k + 1 partial
                if (tid == 0 && k + 2 < nrows) mbar_arrive_expect_tx(rb, xbytes);
            } else {
                if (tid < (int)P) {
                    const uint32_t dst = mapa_shared(smem_u32(&sl[rank * kSlotStride]), (uint32_t)tid);
                    st_cluster_v4f32(dst, p0, p1, p2, 0.f);
                }
                cluster_arrive_release();
                cluster_wait_acquire();
            }
            combine_slots<OP>(sl, P, st0, st1, st2);
        }
        if (tid == 0) {
            const float v[3] = {st0, st1, st2};
            debug_row_stats(a.dbg_stats, row, rank, P, v, 3);
        }

        // a7: apply h to the staged slice; each chunk slot goes back to the
        // producer as soon as this warp's tiles have moved past it, so the
        // next row's copies stream in while this row is still being written
        const OutputMap<OP, T> h(st0, st1, st2, p0, a.cols, a.eps);
        T* yrow = static_cast<T*>(a.y) + row * a.cols + start;
        int released = 0;  // chunks of this row this warp has handed back
        auto release = [&](int next_vec) {
            const int done = min(cpr, next_vec / vpc);
            if (done > released) {
                __syncwarp();
                if (lane == 0)
                    for (int c = released; c < done; ++c)
                        mbar_arrive(smem_u32(&empty_bar[rs * cpr_full + c]));
                released = done;
            }
        };
        output_tiles<OP, T, PT>(h, base, yrow, gp ? gp + start : nullptr, bp ? bp + start : nullptr,
                                nvec, warp, ncw, lane, release);
        release(cpr * vpc);  // chunks past the slice's vectors (none when the slice fills them)
        if (++rs == NR) { rs = 0; ++use; }
    }
    if (clustered && nrows == 0) cluster_wait_acquire();  // entry phase
    if (async_x) {
        // every deposit addressed to this CTA has landed; stay until the
        // whole cluster can say the same
        cluster_arrive_relaxed();
        cluster_wait_acquire();
    }
}

// The warp-specialised form of the same pipeline.  The consumer warps are
// split by role so that a row's reduction overlaps the previous row's output:
//   - reducer warps [0, nred) fold each chunk of row k as it lands, merge the
//     CTA partial (named barrier among themselves), exchange it with st.async
//     deposits, combine the P slots and hand the row's statistics to the
//     storers through a double-buffered hand-off (one "full" mbarrier per
//     buffer, arrived by one reducer thread; one "empty" mbarrier, arrived by
//     every storer warp once it has read the statistics);
//   - storer warps [nred, ncw) wait for row k's statistics, apply h to the
//     staged slice, write it and hand each chunk slot back to the producer as
//     their tiles pass it;
//   - the producer warp streams the rows into the ring as in the kernel above.
// A CTA owns the same column slice of every row it handles, so when the plan
// leaves room for them the storers copy the slice's parameters (gamma / beta,
// weight) into shared memory once per launch and read them from there for
// every row, instead of streaming them from L2 row after row.
// While the storers write row k the reducers are already folding row k + 1
// (its chunks land in the slots the storers have released, or in the next row
// slot when the ring holds two or more rows).  The exchange is always the
// st.async one: only the reducers take part in it, and the cluster barrier is
// met twice (entry and exit) by every warp.
template <int OP, typename T, typename PT>
__global__ void __launch_bounds__(kPersistMaxThreads, 1)
cluster_pipelined(const PersistArgs a) {
    using E = Elem<T>;
    constexpr int VEC = E::kVec;
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(16) float slots[2][kMaxCluster * kSlotStride];
    __shared__ __align__(16) float red[2][2][(kPersistMaxThreads / 32) * 2];  // [row parity][stage]
    __shared__ __align__(16) float hand[2][4];  // row statistics for the storers, by row parity
    __shared__ __align__(8) uint64_t full_bar[kPersistMaxSlots];
    __shared__ __align__(8) uint64_t empty_bar[kPersistMaxSlots];
    __shared__ __align__(8) uint64_t recv_bar[2];     // st.async deposits, by row parity
    __shared__ __align__(8) uint64_t hand_full[2];    // reducers -> storers
    __shared__ __align__(8) uint64_t hand_empty[2];   // storers -> reducers

    const uint32_t P = cluster_nctarank();
    const uint32_t rank = cluster_ctarank();
    const int64_t cid = blockIdx.x / P;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int ncw = (int)(blockDim.x >> 5) - 1;  // reducer + storer warps; the last warp produces
    const int nred = a.reducers;                 // 1 <= nred < ncw (checked by the host)
    const int nsto = ncw - nred;
    const int64_t start = (int64_t)rank * a.slice;
    const int cpr_full = (a.slice + a.chunk - 1) / a.chunk;
    const int NR = a.nslots / cpr_full;
    // checked build: the ring and the parameter room must fit the launch
    const bool fits = layout_fits((uint64_t)a.nslots * a.chunk * sizeof(T), (int64_t)NR * cpr_full,
                                  kPersistMaxSlots, a.err) &&
                      (a.param_off == 0 ||
                       layout_fits((uint64_t)a.param_off + (uint64_t)a.param_room, 0, 0, a.err));
    const int n = fits ? (int)max((int64_t)0, min(a.cols - start, (int64_t)a.slice)) : 0;
    const int nvec = n / VEC;
    const int vpc = a.chunk / VEC;
    const int cpr = (n + a.chunk - 1) / a.chunk;
    const uint32_t ring_s = smem_u32(ring);
    const uint32_t slot_bytes = (uint32_t)a.chunk * (uint32_t)sizeof(T);
    const int64_t nrows = cid < a.rows ? (a.rows - 1 - cid) / a.nclusters + 1 : 0;
    const bool clustered = P > 1;
    const uint32_t xbytes = (P - 1) * 16u;
    // Every wait is bounded; a thread whose wait gave up (the device error
    // word records it) skips its later waits, so a launch that went wrong
    // ends after one time limit per thread instead of one per wait.
    bool live = true;
    auto wait = [&](uint64_t* bar, uint32_t parity) {
        if (live) live = mbar_wait_bounded(smem_u32(bar), parity, a.err);
    };

    if (tid == 0) {
        for (int s = 0; s < (fits ? NR * cpr_full : 0); ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), (uint32_t)nsto);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&hand_full[b]), 1);
            mbar_init(smem_u32(&hand_empty[b]), (uint32_t)nsto);
            if (clustered) {
                mbar_init(smem_u32(&recv_bar[b]), 2);
                if (b < nrows) mbar_arrive_expect_tx(smem_u32(&recv_bar[b]), xbytes);
            }
        }
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    __syncthreads();
    if (clustered) cluster_arrive_relaxed();

    // ------------------------------------------------------------ producer
    if (warp == ncw) {
        const uint64_t pol = l2_policy_evict_first();
        int rs = 0;
        uint32_t use = 0;
        for (int64_t k = 0; k < nrows; ++k) {
            if (lane == 0) {
                const T* src = static_cast<const T*>(a.x) + (cid + k * a.nclusters) * a.cols + start;
                for (int c = 0; c < cpr; ++c) {
                    const int slot = rs * cpr_full + c;
                    if (use > 0) wait(&empty_bar[slot], (use - 1) & 1u);
                    const int e0 = c * a.chunk;
                    const uint32_t bytes = (uint32_t)(min(a.chunk, n - e0) * (int)sizeof(T));
                    const uint32_t fb = smem_u32(&full_bar[slot]);
                    mbar_arrive_expect_tx(fb, bytes);
                    bulk_g2s(ring_s + (uint32_t)slot * slot_bytes, src + e0, bytes, fb, pol);
                }
            }
            if (++rs == NR) { rs = 0; ++use; }
            __syncwarp();
        }
        if (clustered) {
            cluster_wait_acquire();    // entry
            cluster_arrive_relaxed();  // exit
            cluster_wait_acquire();
        }
        return;
    }

    if (warp < nred) {
        // --------------------------------------------------------- reducers
        const int nrt = nred * 32;
        int rs = 0;
        uint32_t use = 0;
        for (int64_t k = 0; k < nrows; ++k) {
            unsigned char* base = ring + (size_t)rs * cpr_full * slot_bytes;
            Stats<OP, T> stt;
            for (int c = 0; c < cpr; ++c) {
                wait(&full_bar[rs * cpr_full + c], use & 1u);
                const int v0 = c * vpc;
                stats_tiles(stt, base + (size_t)v0 * 16, min(nvec, v0 + vpc) - v0, warp, nred, lane);
            }
            auto stash = [&](float mq) { return softmax_stash(base, nvec, warp, nred, lane, mq); };
            float p0, p1, p2;
            cta_partial<OP, T>(stt, red[k & 1][0], red[k & 1][1], nred, nrt, stash, p0, p1, p2);
            // the fp32 softmax stash wrote the slots: order those generic-proxy
            // writes before the bulk copies that will refill them
            if constexpr (OP == kSoftmax && sizeof(T) == 4) fence_proxy_async_smem();

            float st0 = p0, st1 = p1, st2 = p2;
            if (clustered) {
                if (k == 0) cluster_wait_acquire();  // every peer is running
                float* sl = slots[k & 1];
                const uint32_t rb = smem_u32(&recv_bar[k & 1]);
                if (tid == (int)rank) {
                    float* d = &sl[rank * kSlotStride];
                    d[0] = p0; d[1] = p1; d[2] = p2;
                    mbar_arrive(rb);
                } else if (tid < (int)P) {
                    const uint32_t dst = mapa_shared(smem_u32(&sl[rank * kSlotStride]), (uint32_t)tid);
                    st_async_v4f32(dst, p0, p1, p2, 0.f, mapa_shared(rb, (uint32_t)tid));
                }
                wait(&recv_bar[k & 1], (uint32_t)(k >> 1) & 1u);
                // no peer deposits row k + 2 before this CTA's row k + 1
                // partial, which follows this row's combine below
                if (tid == 0 && k + 2 < nrows) mbar_arrive_expect_tx(rb, xbytes);
                combine_slots<OP>(sl, P, st0, st1, st2);
            }
            if (tid == 0) {
                const float v[3] = {st0, st1, st2};
                debug_row_stats(a.dbg_stats, cid + k * a.nclusters, rank, P, v, 3);
                // the hand-off buffer of row k was last read for row k - 2
                if (k >= 2)
                    wait(&hand_empty[k & 1], (uint32_t)((k >> 1) - 1) & 1u);
                float* h = hand[k & 1];
                h[0] = st0; h[1] = st1; h[2] = st2; h[3] = p0;
                mbar_arrive(smem_u32(&hand_full[k & 1]));
            }
            if (++rs == NR) { rs = 0; ++use; }
        }
        if (clustered && nrows == 0) cluster_wait_acquire();  // entry
    } else {
        // ----------------------------------------------------------- storers
        const int sw = warp - nred;
        const PT* gp = static_cast<const PT*>(a.p0);
        const PT* bp = static_cast<const PT*>(a.p1);
        constexpr bool kParams = OP == kLayerNorm || OP == kRMSNorm;
        const int pbytes = (n * (int)sizeof(PT) + 15) & ~15;  // one parameter's slice, padded
        const int need = kParams ? (gp ? pbytes : 0) + (bp ? pbytes : 0) : 0;
        const bool pstage = need > 0 && a.param_off > 0 && need <= a.param_room;
        const PT* gs = nullptr;
        const PT* bs = nullptr;
        if (pstage) {
            // the storers copy the slice's parameters into the room once
            unsigned char* room = ring + a.param_off;
            const int stid = tid - nred * 32, nst = nsto * 32;
            auto copy_slice = [&](const PT* src, unsigned char* dst) {
                const PT* s0 = src + start;
                int done = 0;
                if ((reinterpret_cast<uintptr_t>(s0) & 15) == 0) {
                    const int nv = n * (int)sizeof(PT) / 16;
                    for (int i = stid; i < nv; i += nst)
                        reinterpret_cast<uint4*>(dst)[i] = __ldg(reinterpret_cast<const uint4*>(s0) + i);
                    done = nv * 16 / (int)sizeof(PT);
                }
                for (int i = done + stid; i < n; i += nst) reinterpret_cast<PT*>(dst)[i] = s0[i];
            };
            if (gp) { copy_slice(gp, room); gs = reinterpret_cast<const PT*>(room); }
            if (bp) {
                unsigned char* d = room + (gp ? pbytes : 0);
                copy_slice(bp, d);
                bs = reinterpret_cast<const PT*>(d);
            }
            named_sync_id(2, nst);  // the storers only
        }
        if (clustered) cluster_wait_acquire();  // entry
        int rs = 0;
        uint32_t use = 0;
        for (int64_t k = 0; k < nrows; ++k) {
            const int64_t row = cid + k * a.nclusters;
            unsigned char* base = ring + (size_t)rs * cpr_full * slot_bytes;
            wait(&hand_full[k & 1], (uint32_t)(k >> 1) & 1u);
            const float* h4 = hand[k & 1];
            const float st0 = h4[0], st1 = h4[1], st2 = h4[2], mq = h4[3];
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&hand_empty[k & 1]));
            // the slice's copies have completed (the reducers waited for them
            // before the hand-off); observe their phases here as well
            for (int c = 0; c < cpr; ++c)
                wait(&full_bar[rs * cpr_full + c], use & 1u);
            const OutputMap<OP, T> hm(st0, st1, st2, mq, a.cols, a.eps);
            T* yrow = static_cast<T*>(a.y) + row * a.cols + start;
            int released = 0;
            auto release = [&](int next_vec) {
                const int done = min(cpr, next_vec / vpc);
                if (done > released) {
                    __syncwarp();
                    if (lane == 0)
                        for (int c = released; c < done; ++c)
                            mbar_arrive(smem_u32(&empty_bar[rs * cpr_full + c]));
                    released = done;
                }
            };
            if (pstage) {
                output_tiles<OP, T, PT, decltype(release), true>(hm, base, yrow, gs, bs, nvec, sw,
                                                                 nsto, lane, release);
            } else {
                output_tiles<OP, T, PT>(hm, base, yrow, gp ? gp + start : nullptr,
                                        bp ? bp + start : nullptr, nvec, sw, nsto, lane, release);
            }
            release(cpr * vpc);
            if (++rs == NR) { rs = 0; ++use; }
        }
    }
    if (clustered) {
        // every deposit addressed to this CTA has landed (the reducers waited
        // for each row's); stay until the whole cluster can say the same
        cluster_arrive_relaxed();
        cluster_wait_acquire();
    }
}

// ----------------------------------------------------------- dispatch
template <int OP, typename T>
static const void* pers_param(int pdtype) {
    return pdtype == 0 ? (const void*)cluster_persistent<OP, T, float>
                       : (const void*)cluster_persistent<OP, T, bf16>;
}

template <int OP, typename T>
static const void* pipe_param(int pdtype) {
    return pdtype == 0 ? (const void*)cluster_pipelined<OP, T, float>
                       : (const void*)cluster_pipelined<OP, T, bf16>;
}

const void* pipelined_kernel(KernelKey k) {
    if (!k.vec) return nullptr;
    switch (k.op) {
        case kSoftmax: return k.dtype == 0 ? (const void*)cluster_pipelined<kSoftmax, float, float>
                                           : (const void*)cluster_pipelined<kSoftmax, bf16, float>;
        case kLayerNorm: return k.dtype == 0 ? pipe_param<kLayerNorm, float>(k.pdtype)
                                             : pipe_param<kLayerNorm, bf16>(k.pdtype);
        case kRMSNorm: return k.dtype == 0 ? pipe_param<kRMSNorm, float>(k.pdtype)
                                           : pipe_param<kRMSNorm, bf16>(k.pdtype);
    }
    return nullptr;
}

// Reducer / storer split of the warp-specialised kernel, from the relative
// per-element work of the two roles: softmax recomputes the exponential in
// both (bf16) or stashes it in the reduction (fp32); the norms' output pass
// carries the parameter loads, RMSNorm's reduction is one FMA per element.
int pipelined_reducers(int op, int dtype, int consumer_warps) {
    int r = consumer_warps / 2;
    if (op == kSoftmax && dtype == 0) r = (consumer_warps * 5) / 8;
    if (op == kLayerNorm) r = (consumer_warps * 3) / 8;
    if (op == kRMSNorm) r = consumer_warps / 4;
    return max(1, min(consumer_warps - 1, r));
}

const void* persistent_kernel(KernelKey k) {
    if (!k.vec) return nullptr;  // the ring is filled by bulk copies only
    switch (k.op) {
        case kSoftmax: return k.dtype == 0 ? (const void*)cluster_persistent<kSoftmax, float, float>
                                           : (const void*)cluster_persistent<kSoftmax, bf16, float>;
        case kLayerNorm: return k.dtype == 0 ? pers_param<kLayerNorm, float>(k.pdtype)
                                             : pers_param<kLayerNorm, bf16>(k.pdtype);
        case kRMSNorm: return k.dtype == 0 ? pers_param<kRMSNorm, float>(k.pdtype)
                                           : pers_param<kRMSNorm, bf16>(k.pdtype);
    }
    return nullptr;
}

cudaError_t launch_persistent(KernelKey k, const PersistArgs& a, int P, int threads,
                              size_t smem, cudaStream_t s) {
    const void* fn = a.reducers > 0 ? pipelined_kernel(k) : persistent_kernel(k);
    if (!fn) return cudaErrorInvalidDeviceFunction;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.nclusters * P), 1, 1);
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
    PersistArgs b = a;
    void* args[] = {&b};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace credit
