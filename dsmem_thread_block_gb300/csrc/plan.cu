// plan.cu -- plan legality and candidate selection.
//
// Legality (CREDIT summary page, arXiv 2609.01864v1, "B. Reduction-Reuse
// Transformation", resource constraint): a cluster size P is legal when the
// retained slice (ceil(N / P) elements rounded up to a 16-byte vector, times
// the element size) plus the kernel's fixed per-CTA scratch fits the
// dynamic-shared-memory opt-in limit, and the device can keep at least one
// such cluster resident (cudaOccupancyMaxActiveClusters; clusters must fit
// in one GPC, so the page's floor(S / P) is replaced by the runtime's count).
#include <algorithm>
#include <cmath>
#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "planner.h"

namespace credit {

namespace {

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

bool op_ok(credit_op_t op) {
    return op == CREDIT_SOFTMAX || op == CREDIT_LAYERNORM || op == CREDIT_RMSNORM ||
           op == CREDIT_QUANTIZE || op == CREDIT_WEIGHTED_STD || op == CREDIT_PEARSON;
}

int cluster_threads(int64_t staged_vecs) {
    // about sixteen 16-byte vectors per thread (four warp tiles of four), warp
    // multiples, 64..256 threads: three such CTAs share an SM
    int64_t t = round_up(std::max<int64_t>(1, staged_vecs / 16), 32);
    return (int)std::min<int64_t>(256, std::max<int64_t>(64, t));
}

// Static model used until the device is calibrated: one HBM stream at a
// nominal rate, derated when fewer than two CTAs share an SM (nothing hides
// a CTA's load -> reduce -> barrier -> store sequence), plus a fixed cost per
// wave of resident clusters.
constexpr double kNominalBytesPerUs = 6.0e6;
constexpr double kWaveUsCluster = 1.5;
constexpr double kWaveUsSingle = 0.5;
constexpr double kLaunchUs = 3.0;

}  // namespace

int64_t bulk_chunk_elems(int64_t slice_elems, int elem_bytes, int rows_per_cluster) {
    const int64_t vec = 16 / elem_bytes;
    const int64_t target = 16384 / elem_bytes;
    return round_up(std::max(target, ceil_div(slice_elems, kMaxChunks / rows_per_cluster)), vec);
}

bool deep_footprint(int dev, KernelKey k, int64_t smem_bytes) {
    const DevInfo* d = device_info(dev);
    k.deep = false;
    const KernelInfo* ki = d ? kernel_info(dev, cluster_kernel(k), true) : nullptr;
    if (!ki) return false;
    return smem_bytes + ki->static_smem + d->reserved_smem > (int64_t)d->smem_per_sm / 3;
}

bool quad_footprint(int dev, KernelKey k, int64_t smem_bytes, bool tail) {
    if (!tail || !k.vec || k.rows != 1 ||
        !quad_capable(k.op, k.dtype == 0 ? 4 : 2, k.pdtype == 1 ? 2 : 4))
        return false;
    const DevInfo* d = device_info(dev);
    k.deep = false;
    k.quad = false;
    const KernelInfo* ki = d ? kernel_info(dev, cluster_kernel(k), true) : nullptr;
    if (!ki) return false;
    return smem_bytes + ki->static_smem + d->reserved_smem <= (int64_t)d->smem_per_sm / 4;
}

int64_t tail_budget_bytes(const DevInfo& d, int static_smem, int cps) {
    const int64_t per_cta = (int64_t)d.smem_per_sm / cps - d.reserved_smem;
    const int64_t kb = 1024;
    return per_cta / kb * kb - (static_smem + kb - 1) / kb * kb - kb;
}

int64_t cluster_slice(int64_t cols, int P, int es) {
    return round_up(ceil_div(cols, P), 128 / es);
}

int64_t tail_staged_for(int dev, credit_op_t op, int64_t cols, credit_dtype_t dtype, int P,
                        int cps, int rows_per_cluster) {
    const int es = dtype == CREDIT_F32 ? 4 : 2;
    const int R = rows_per_cluster;
    if (P < 1 || P > kMaxCluster || cps < 1 || (R != 1 && R != 2 && R != 4) ||
        !tail_capable((int)op, es))
        return 0;
    const DevInfo* d = device_info(dev);
    const void* fn = cluster_kernel(KernelKey{(int)op, (int)dtype, 0, true, R});
    const KernelInfo* ki = d ? kernel_info(dev, fn, true) : nullptr;
    if (!ki) return 0;
    const int64_t vec = 16 / es;
    const int64_t slice = cluster_slice(cols, P, es);
    const int64_t budget = std::min<int64_t>(tail_budget_bytes(*d, ki->static_smem, cps),
                                             ki->max_dyn_smem);
    // one row: whole 16-byte vectors; several rows: each staged slice
    // starts on a 128-byte pitch
    const int64_t held = R == 1 ? budget / (vec * es) * vec : budget / R / 128 * 128 / es;
    return held >= vec && held < slice ? held : 0;
}

int64_t row_pitch(int64_t slice_elems, int elem_bytes) {
    return round_up(slice_elems * elem_bytes, 128);
}

namespace {

// Persistent plan for a given (P, CTAs per SM).
credit_status_t persistent_plan(int dev, const DevInfo* d, credit_op_t op, int64_t rows,
                                int64_t cols, credit_dtype_t dtype, int P, int threads,
                                int cps, int64_t chunk_override, bool pipelined,
                                credit_plan_t* p) {
    const int es = dtype == CREDIT_F32 ? 4 : 2;
    const int64_t vec = 16 / es;
    const int64_t slice = round_up(ceil_div(cols, P), vec);
    if (slice > INT32_MAX / 4) return CREDIT_ERR_NO_LEGAL_PLAN;
    // a slot holds a power-of-two number of 16-byte vectors: 16 KiB, or the
    // next power of two above a smaller slice (one slot per row then)
    int64_t chunk_vecs = 16384 / 16;
    if (chunk_override > 0) chunk_vecs = chunk_override / vec;
    if (chunk_vecs < 1 || (chunk_vecs & (chunk_vecs - 1)) != 0 || chunk_vecs * 16 > (1 << 20))
        return CREDIT_ERR_INVALID_ARG;
    while (chunk_vecs / 2 * vec >= slice) chunk_vecs /= 2;
    const int64_t chunk = chunk_vecs * vec;
    const int64_t chunk_bytes = chunk * es;
    const int64_t cpr = ceil_div(slice, chunk);
    const KernelKey key{(int)op, (int)dtype, 0, true};
    const void* fn = pipelined ? pipelined_kernel(key) : persistent_kernel(key);
    if (!fn) return CREDIT_ERR_NO_LEGAL_PLAN;  // operator not offered by the persistent kernel
    const KernelInfo* ki = kernel_info(dev, fn, true);
    if (!ki) return CREDIT_ERR_CUDA;
    const int64_t budget = cps == 1
        ? ki->max_dyn_smem
        : (int64_t)d->smem_per_sm / cps - ki->static_smem - d->reserved_smem;
    // the warp-specialised kernel keeps the slice's parameters in shared
    // memory when a room for them (fp32-sized, else sized like the data
    // elements) fits beside two row slots of the ring, one CTA per SM (with
    // one row slot the next row's reduction waits for this row's output,
    // which costs more than the parameter stream saves)
    int64_t room = 0;
    if (pipelined && cps == 1 && (op == CREDIT_LAYERNORM || op == CREDIT_RMSNORM)) {
        const int np = op == CREDIT_LAYERNORM ? 2 : 1;
        for (int pes : {4, es}) {
            const int64_t r = np * round_up(slice * pes, 16);
            if (2 * cpr * chunk_bytes + r <= budget) {
                room = r;
                break;
            }
        }
    }
    const int64_t fit = std::min<int64_t>(kPersistMaxSlots, (budget - room) / chunk_bytes);
    // the ring holds whole row slices (contiguous in shared memory): at least
    // one, up to three
    const int64_t nr = std::min<int64_t>(3, fit / cpr);
    if (nr < 1) return CREDIT_ERR_NO_LEGAL_PLAN;  // a whole slice must fit the ring
    const int64_t S = nr * cpr;
    const int t = threads ? threads : (cps == 1 ? kPersistMaxThreads : 288);
    // one producer warp plus at least one consumer warp (one reducer and one
    // storer warp in the warp-specialised form)
    if (t < (pipelined ? 96 : 64) || t > kPersistMaxThreads) return CREDIT_ERR_INVALID_ARG;
    const int64_t smem = S * chunk_bytes + room;  // the ring, then the parameter room
    const int active = occupancy_clusters(dev, fn, P, t, (size_t)smem, rows);
    if (active < 1) return CREDIT_ERR_NO_LEGAL_PLAN;
    const int64_t G = std::min<int64_t>(active, rows);
    p->variant = pipelined ? CREDIT_CLUSTER_PIPELINED : CREDIT_CLUSTER_PERSISTENT;
    p->cluster_size = P;
    p->threads = t;
    p->smem_bytes = smem;
    p->slice_elems = slice;
    p->chunk_elems = (int32_t)chunk;
    p->ring_slots = (int32_t)S;
    p->active_clusters = (int32_t)G;
    p->ctas_per_sm = cps;
    p->rows_per_cluster = 1;
    p->exchange = CREDIT_EXCHANGE_ASYNC;
    p->waves = (int32_t)std::min<int64_t>(ceil_div(rows, G), INT32_MAX);
    const double bytes = (op == CREDIT_PEARSON ? 3.0 : 2.0) * (double)rows * (double)cols * es;
    const double coverage = std::min(1.0, (double)G * P / ((double)d->sms * cps));
    const double pipe = nr >= 2 ? 0.95 : 0.8;
    p->pred_us = (float)(bytes / (kNominalBytesPerUs * coverage * pipe) + kLaunchUs);
    return CREDIT_OK;
}

}  // namespace

credit_status_t make_plan(int dev, credit_op_t op, int64_t rows, int64_t cols,
                          credit_dtype_t dtype, credit_variant_t variant, int P,
                          int threads, int cps, credit_plan_t* out, int64_t chunk,
                          int rows_per_cluster, int64_t staged_req) {
    if (!out || rows < 1 || cols < 1) return CREDIT_ERR_INVALID_ARG;
    if (!op_ok(op)) return CREDIT_ERR_UNSUPPORTED;
    if (dtype != CREDIT_F32 && dtype != CREDIT_BF16) return CREDIT_ERR_UNSUPPORTED;
    if (threads != 0 && (threads < 32 || threads % 32 != 0)) return CREDIT_ERR_INVALID_ARG;
    const bool ring = variant == CREDIT_CLUSTER_PERSISTENT || variant == CREDIT_CLUSTER_PIPELINED;
    if (threads > (ring ? kPersistMaxThreads
                   : variant == CREDIT_CLUSTER             ? kClusterMaxThreads
                                                           : kMaxThreads))
        return CREDIT_ERR_INVALID_ARG;
    const DevInfo* d = device_info(dev);
    if (!d) return CREDIT_ERR_CUDA;
    const int es = dtype == CREDIT_F32 ? 4 : 2;
    const int64_t vec = 16 / es;
    credit_plan_t p;
    std::memset(&p, 0, sizeof(p));
    p.variant = variant;
    p.ctas_per_sm = 1;
    // st.async deposits for both clustered kernels (measured faster than
    // the push + barrier exchange in each)
    p.exchange = (variant == CREDIT_TWO_PASS || variant == CREDIT_WARP_ROWS)
                     ? CREDIT_EXCHANGE_DEFAULT : CREDIT_EXCHANGE_ASYNC;
    const double bytes = (op == CREDIT_PEARSON ? 3.0 : 2.0) * (double)rows * (double)cols * es;

    if (variant == CREDIT_CLUSTER) {
        if (P < 1 || P > kMaxCluster) return CREDIT_ERR_NO_LEGAL_PLAN;
        const int R = rows_per_cluster ? rows_per_cluster : 1;
        if (R != 1 && R != 2 && R != 4) return CREDIT_ERR_INVALID_ARG;
        // Pearson stages two operands (x, then u one pitch further) of one row
        const bool two_ops = op == CREDIT_PEARSON;
        if (two_ops && R != 1) return CREDIT_ERR_INVALID_ARG;
        const int staged = two_ops ? 2 : R;  // slices held per CTA
        const int64_t slice = cluster_slice(cols, P, es);
        // an L2 tail: stage only the first `held` elements of each row's
        // slice (operators without an in-place stash pass)
        int64_t held = slice;
        if (staged_req > 0 && staged_req < slice) {
            if (two_ops || !tail_capable((int)op, es)) return CREDIT_ERR_INVALID_ARG;
            held = round_up(staged_req, vec);
        }
        const int64_t pitch = row_pitch(held, es);
        const int64_t smem = staged == 1 ? round_up(held * es, 16) : staged * pitch;
        KernelKey key{(int)op, (int)dtype, 0, true, R};
        key.quad = quad_footprint(dev, key, smem, held < slice);
        const void* fn = cluster_kernel(key);
        const KernelInfo* ki = kernel_info(dev, fn, true);
        if (!ki) return CREDIT_ERR_CUDA;
        if (smem > ki->max_dyn_smem || pitch > INT32_MAX) return CREDIT_ERR_NO_LEGAL_PLAN;
        const int t = threads ? threads : cluster_threads(staged * slice / vec);
        const int active = occupancy_clusters(dev, fn, P, t, (size_t)smem, rows);
        if (active < 1) return CREDIT_ERR_NO_LEGAL_PLAN;
        p.cluster_size = P;
        p.threads = t;
        p.smem_bytes = smem;
        p.slice_elems = slice;
        p.staged_elems = held;
        p.chunk_elems = (int32_t)bulk_chunk_elems(held, es, staged);
        p.rows_per_cluster = R;
        p.active_clusters = active;
        p.ctas_per_sm = std::max(1, (int)((int64_t)active * P / d->sms));
        p.waves = (int32_t)std::min<int64_t>(ceil_div(ceil_div(rows, R), active), INT32_MAX);
        const double ctas_per_sm = (double)active * P / d->sms;
        const double eff = ctas_per_sm >= 2.0 ? 0.9 : 0.7;
        p.pred_us = (float)(bytes / (kNominalBytesPerUs * eff) +
                            p.waves * (P > 1 ? kWaveUsCluster : kWaveUsSingle));
    } else if (ring) {
        if (P < 1 || P > kMaxCluster) return CREDIT_ERR_NO_LEGAL_PLAN;
        if (cps != 0 && cps != 1 && cps != 2) return CREDIT_ERR_INVALID_ARG;
        credit_status_t best = CREDIT_ERR_NO_LEGAL_PLAN;
        for (int c = 1; c <= 2; ++c) {
            if (cps && c != cps) continue;
            credit_plan_t q;
            std::memset(&q, 0, sizeof(q));
            const credit_status_t st =
                persistent_plan(dev, d, op, rows, cols, dtype, P, threads, c, chunk,
                                variant == CREDIT_CLUSTER_PIPELINED, &q);
            if (st == CREDIT_ERR_CUDA || st == CREDIT_ERR_INVALID_ARG) return st;
            if (st == CREDIT_OK && (best != CREDIT_OK || q.pred_us < p.pred_us)) {
                p = q;
                best = CREDIT_OK;
            }
        }
        if (best != CREDIT_OK) return best;
    } else if (variant == CREDIT_WARP_ROWS) {
        // one warp per row, the row in registers: whole rows of at most
        // 32 lanes x kWarpRowNV vectors
        if (ceil_div(cols, vec) > 32 * kWarpRowNV) return CREDIT_ERR_NO_LEGAL_PLAN;
        const void* fn = warp_rows_kernel(KernelKey{(int)op, (int)dtype, 0, true}, ceil_div(cols, vec));
        if (!fn) return CREDIT_ERR_NO_LEGAL_PLAN;  // operator not offered
        if (!kernel_info(dev, fn, false)) return CREDIT_ERR_CUDA;
        const int per_sm = occupancy_clusters(dev, fn, 1, kWarpRowThreads, 0, rows);
        if (per_sm < 1) return CREDIT_ERR_NO_LEGAL_PLAN;
        const int64_t wpb = kWarpRowThreads / 32;
        const int64_t blocks = std::min<int64_t>(per_sm, ceil_div(rows, wpb));
        p.cluster_size = 1;
        p.threads = kWarpRowThreads;
        p.slice_elems = cols;
        p.active_clusters = (int32_t)blocks;
        p.rows_per_cluster = 1;
        p.waves = (int32_t)std::min<int64_t>(ceil_div(rows, blocks * wpb), INT32_MAX);
        p.pred_us = (float)(bytes / (kNominalBytesPerUs * 0.9) + kLaunchUs);
    } else if (variant == CREDIT_TWO_PASS) {
        const int64_t per_thread = kTwoPassVpt * vec;
        int t = threads;
        if (!t) {
            t = cols >= (int64_t)kMaxThreads * per_thread
                    ? kMaxThreads
                    : (int)std::max<int64_t>(32, round_up(ceil_div(cols, per_thread), 32));
        }
        const int64_t chunk = (int64_t)t * per_thread;
        const int64_t nch = ceil_div(cols, chunk);
        if (nch > INT32_MAX) return CREDIT_ERR_INVALID_ARG;
        const void* fn = two_pass_stats_kernel(KernelKey{(int)op, (int)dtype, 0, true});
        const KernelInfo* ki = kernel_info(dev, fn, false);
        if (!ki) return CREDIT_ERR_CUDA;
        const int active = occupancy_clusters(dev, fn, 1, t, 0, rows);
        if (active < 1) return CREDIT_ERR_NO_LEGAL_PLAN;
        p.cluster_size = 1;
        p.rows_per_cluster = 1;
        p.threads = t;
        p.slice_elems = chunk;
        p.chunk_elems = (int32_t)chunk;
        p.workspace_bytes = rows * nch * (op == CREDIT_PEARSON ? 8 : 4) * (int64_t)sizeof(float);
        p.active_clusters = active;
        p.waves = (int32_t)std::min<int64_t>(ceil_div(rows * nch, active), INT32_MAX);
        p.pred_us = (float)(1.5 * bytes / (kNominalBytesPerUs * 0.9) + 2 * kLaunchUs);
        p.pred_two_pass_us = p.pred_us;
    } else {
        return CREDIT_ERR_INVALID_ARG;
    }
    *out = p;
    return CREDIT_OK;
}

credit_status_t auto_plan(int dev, credit_op_t op, int64_t rows, int64_t cols,
                          credit_dtype_t dtype, credit_plan_t* out) {
    if (!out || rows < 1 || cols < 1) return CREDIT_ERR_INVALID_ARG;
    if (forced_plan(dev, op, rows, cols, dtype, out)) return CREDIT_OK;  // CREDIT_FORCE
    credit_plan_t profiled;
    if (lookup_profiled_plan(dev, op, rows, cols, dtype, &profiled)) {
        *out = profiled;
        return CREDIT_OK;
    }
    credit_plan_t base;
    credit_status_t st = make_plan(dev, op, rows, cols, dtype, CREDIT_TWO_PASS, 0, 0, 0, &base);
    if (st != CREDIT_OK) return st;
    // Static choice (no profile for this shape): rows of 2 KiB or less one
    // warp each in registers (softmax, LayerNorm, RMSNorm; measured 1.5x the
    // staging kernel for 1024-column bf16 softmax and LayerNorm rows); else the
    // one-row-per-cluster kernel with the smallest P whose slice stays within
    // 64 KiB (three 256-thread CTAs per SM), rows of 16 KiB or less batched
    // four to a CTA;
    // the two-pass kernel only when no cluster size fits.
    const int es = dtype == CREDIT_F32 ? 4 : 2;
    const int nops = op == CREDIT_PEARSON ? 2 : 1;  // staged operands per row
    if (cols * es <= 2048 && (cols * es) % 16 == 0) {
        credit_plan_t w;
        if (make_plan(dev, op, rows, cols, dtype, CREDIT_WARP_ROWS, 1, 0, 0, &w) == CREDIT_OK) {
            w.pred_two_pass_us = base.pred_us;
            *out = w;
            return CREDIT_OK;
        }
    }
    for (int P = 1; P <= kMaxCluster; ++P) {
        const int64_t slice_bytes = ceil_div(cols, P) * es * nops;
        if (slice_bytes > 65536 && P < kMaxCluster) continue;
        const int R = (P == 1 && nops == 1 && slice_bytes * 4 <= 65536) ? 4 : 1;
        credit_plan_t c;
        if (make_plan(dev, op, rows, cols, dtype, CREDIT_CLUSTER, P, 0, 0, &c, 0, R) != CREDIT_OK)
            continue;
        c.pred_two_pass_us = base.pred_us;
        *out = c;
        return CREDIT_OK;
    }
    base.pred_two_pass_us = base.pred_us;
    *out = base;
    return CREDIT_OK;
}

}  // namespace credit
