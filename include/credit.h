/*
 * credit.h -- C ABI of libcredit: CREDIT's DSMEM reduction-reuse
 * transformation for wide-row reduce-then-reuse operators (row softmax,
 * LayerNorm, RMSNorm, int8 quantization, weighted standardization, Pearson
 * correlation) on GB300 (sm_103a).
 *
 * Operation (CREDIT summary page, arXiv 2609.01864v1, "B. Reduction-Reuse
 * Transformation" and "C. Cluster Reduction and Reuse Protocol"): each row is
 * split into P contiguous slices owned by the P CTAs of one thread-block
 * cluster.  Every CTA stages its slice in shared memory once, reduces it to a
 * compact partial statistic, pushes that partial into a slot that each peer
 * CTA owns (distributed shared memory) -- by default as st.async deposits
 * that complete on the receiver's mbarrier, or with remote stores and a
 * cluster barrier -- combines the P slots with local reads only, and writes
 * its output slice straight from shared memory.  The row is read from HBM
 * once and written once.
 * The non-clustered two-pass kernel (partials to a global workspace, then a
 * second kernel that re-reads the row) ships alongside as the in-library
 * baseline ("A. Experimental Setup and Baselines": a non-DSMEM CUDA baseline
 * that either stages locally or re-reads global memory).
 *
 * Conventions for every entry point:
 *  - Pointers named x, u, y, q, scales, r, gamma, beta, weight(s), workspace
 *    are DEVICE pointers on the current CUDA device; the caller owns them.
 *    Nothing on the call path allocates memory.  (credit_run_host takes host
 *    buffers; the calibration and microbenchmark calls allocate scratch.)
 *  - Matrices are row-major with row stride == cols (contiguous rows).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Calls are asynchronous on that stream and never synchronise
 *    the host; a launch error is returned as CREDIT_ERR_CUDA.
 *  - y == x (in place) is allowed; any other overlap of x and y is rejected.
 *  - Errors are returned as credit_status_t; nothing is thrown.
 *  - Calls are thread-safe.  The only state is a per-device cache of kernel
 *    attributes and of the calibration profile.
 */
#ifndef CREDIT_H
#define CREDIT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CREDIT_OK = 0,
    CREDIT_ERR_INVALID_ARG = 1,     /* null / overlapping / misaligned / bad size */
    CREDIT_ERR_UNSUPPORTED = 2,     /* dtype or op not supported */
    CREDIT_ERR_NO_LEGAL_PLAN = 3,   /* forced plan breaks the SMEM legality rule */
    CREDIT_ERR_CUDA = 4,            /* a CUDA runtime call failed */
    CREDIT_ERR_DEVICE_TIMEOUT = 5,  /* a bounded device-side wait gave up */
    CREDIT_ERR_NOT_CALIBRATED = 6,  /* the cost model has no profile yet */
    CREDIT_ERR_DEVICE_BOUNDS = 7    /* checked build: a device index check failed */
} credit_status_t;

typedef enum { CREDIT_F32 = 0, CREDIT_BF16 = 1 } credit_dtype_t;

typedef enum {
    CREDIT_SOFTMAX = 0,
    CREDIT_LAYERNORM = 1,
    CREDIT_RMSNORM = 2,
    CREDIT_QUANTIZE = 3,      /* row absmax -> scale -> int8 codes */
    CREDIT_WEIGHTED_STD = 4,  /* weighted standardization, per-column weights */
    CREDIT_PEARSON = 5        /* row correlation of two matrices, co-deviations out */
} credit_op_t;

typedef enum {
    CREDIT_AUTO = 0,       /* let credit_plan decide */
    CREDIT_CLUSTER = 1,    /* clustered DSMEM kernel, one row per cluster of
                              cluster_size = P CTAs (1..16) */
    CREDIT_TWO_PASS = 2,   /* non-clustered two-pass re-read kernel pair */
    CREDIT_CLUSTER_PERSISTENT = 3, /* clustered DSMEM kernel, resident clusters
                              loop over rows; a producer warp streams chunks
                              into a ring of shared-memory slots */
    CREDIT_CLUSTER_PIPELINED = 4,  /* the persistent kernel with warp-specialised
                              consumers: reducer warps fold, exchange and
                              combine row k + 1 while storer warps write row
                              k (softmax, LayerNorm, RMSNorm; ASYNC exchange
                              only) */
    CREDIT_WARP_ROWS = 5           /* non-clustered: one warp holds a whole row
                              in registers (rows of at most 4 KiB; softmax,
                              LayerNorm, RMSNorm; no exchange) */
} credit_variant_t;

/*
 * How the clustered kernels hand their partials to the peers
 * (credit_plan_t.exchange):
 *   DEFAULT  in a request: let the planner choose; in a planned TWO_PASS
 *            plan: there is no exchange
 *   BARRIER  remote 16-byte stores into every peer's slot array, then a
 *            release/acquire cluster barrier (CREDIT "C. Cluster Reduction
 *            and Reuse Protocol", Replicated Push + Synchronization)
 *   ASYNC    st.async 16-byte deposits whose bytes complete on the receiving
 *            CTA's mbarrier; each CTA waits for its own P - 1 deposits, and
 *            the cluster barrier moves to kernel exit (the planner's choice
 *            for both clustered variants; the persistent kernel alternates
 *            two mbarriers by row parity)
 */
typedef enum {
    CREDIT_EXCHANGE_DEFAULT = 0,
    CREDIT_EXCHANGE_BARRIER = 1,
    CREDIT_EXCHANGE_ASYNC = 2
} credit_exchange_t;

/*
 * A launch plan.  Produced by credit_plan / credit_plan_for; may be passed to
 * the operator calls (NULL there means "plan automatically").
 *   variant          CREDIT_CLUSTER, CREDIT_CLUSTER_PERSISTENT,
 *                    CREDIT_CLUSTER_PIPELINED, CREDIT_WARP_ROWS or
 *                    CREDIT_TWO_PASS (never AUTO once planned); WARP_ROWS
 *                    plans have cluster_size 1, smem_bytes 0 and
 *                    active_clusters = the CTAs of their row-striding grid
 *   cluster_size     P, CTAs per row (1..16; 1 = one CTA stages the whole row)
 *   threads          threads per CTA
 *   waves            predicted waves of resident clusters, ceil(rows / active)
 *   smem_bytes       dynamic shared memory per CTA (staged slice or ring)
 *   workspace_bytes  device workspace the call needs (TWO_PASS only, else 0)
 *   slice_elems      elements of a row owned by one CTA (CLUSTER variants) or
 *                    one chunk (TWO_PASS)
 *   active_clusters  clusters resident at once (cudaOccupancyMaxActiveClusters);
 *                    the persistent grid has this many clusters
 *   ctas_per_sm      CTAs the plan expects to share one SM
 *   chunk_elems      elements per bulk copy (one mbarrier each)
 *   ring_slots       shared-memory chunk slots per CTA (persistent and
 *                    pipelined only)
 *   rows_per_cluster rows one cluster stages and reduces together (CLUSTER:
 *                    1, 2 or 4; their partials share one exchange and each
 *                    parameter load serves all of them)
 *   exchange         credit_exchange_t: ASYNC for planned clustered plans,
 *                    DEFAULT for TWO_PASS; a request may ask for BARRIER on
 *                    either clustered variant
 *   pred_us          predicted time of this plan, microseconds (0 = none)
 *   pred_two_pass_us predicted / measured time of the two-pass baseline
 */
typedef struct {
    int32_t variant;
    int32_t cluster_size;
    int32_t threads;
    int32_t waves;
    int64_t smem_bytes;
    int64_t workspace_bytes;
    int64_t slice_elems;
    int32_t active_clusters;
    int32_t ctas_per_sm;
    int32_t chunk_elems;
    int32_t ring_slots;
    int32_t rows_per_cluster;
    int32_t exchange;
    float pred_us;
    float pred_two_pass_us;
    int64_t staged_elems;    /* CREDIT_CLUSTER, one row per cluster: elements of
                                each CTA's slice staged in shared memory; the
                                rest of the slice (the L2 tail) is read from
                                HBM once with an L2 evict-last hint, folded
                                from registers, and read again from L2 by the
                                output pass.  In a request it asks for an
                                L2 tail when it lies below the request's own
                                slice_elems, or when slice_elems is 0 (a
                                fresh request); 0, or a value equal to
                                slice_elems (a whole-slice plan as derived),
                                stages the whole slice. */
} credit_plan_t;

/*
 * Plan an operator call automatically (CREDIT "D. Profitability and Candidate
 * Selection": enumerate the legal cluster sizes -- retained slice plus fixed
 * scratch must fit the dynamic-SMEM limit ("B. ... Resource Constraint") --
 * predict each one's time and the two-pass baseline's, and keep the fastest).
 * Uses the calibration profile of `device` if credit_calibrate has run on it,
 * else a static bandwidth model.  Host only; does not launch kernels.
 * Returns CREDIT_ERR_INVALID_ARG for rows < 1, cols < 1 or a null `out`.
 */
credit_status_t credit_plan(credit_op_t op, int64_t rows, int64_t cols,
                            credit_dtype_t dtype, int device,
                            credit_plan_t *out);

/*
 * The L2-tail plan of a one-row-per-cluster launch with cluster size
 * cluster_size whose staged part lets ctas_per_sm (1..32) CTAs share an SM:
 * staged_elems is the largest whole number of 16-byte vectors of the slice
 * that fits that share of an SM's shared memory (how many CTAs are then
 * resident also depends on threads and registers).  CREDIT_ERR_NO_LEGAL_PLAN
 * if the whole slice already fits that budget, the operator and dtype have
 * no L2-tail form (fp32 softmax, quantization, weighted standardization,
 * Pearson), or no such cluster can be resident.  Host only.
 */
credit_status_t credit_plan_tail(credit_op_t op, int64_t rows, int64_t cols,
                                 credit_dtype_t dtype, int device, int cluster_size,
                                 int ctas_per_sm, credit_plan_t *out);

/*
 * Build a plan for a forced variant: CREDIT_CLUSTER, CREDIT_CLUSTER_PERSISTENT
 * or CREDIT_CLUSTER_PIPELINED with the given cluster_size (1..16), or
 * CREDIT_WARP_ROWS / CREDIT_TWO_PASS (cluster_size ignored).
 * Returns CREDIT_ERR_NO_LEGAL_PLAN if the slice does not fit in shared memory
 * or no cluster of that size can be resident.
 */
credit_status_t credit_plan_for(credit_op_t op, int64_t rows, int64_t cols,
                                credit_dtype_t dtype, int device,
                                credit_variant_t variant, int cluster_size,
                                credit_plan_t *out);

/*
 * Complete a plan from a partial request: `request->variant` (CLUSTER,
 * CLUSTER_PERSISTENT, CLUSTER_PIPELINED, WARP_ROWS or TWO_PASS) and, for the
 * clustered variants,
 * `request->cluster_size` are required; `threads`, `ctas_per_sm`,
 * `chunk_elems` and `rows_per_cluster` are used when non-zero and chosen
 * otherwise; every other field is ignored.  The operator calls re-derive a
 * passed plan the same way, so a plan can never launch an illegal shape.
 * Returns CREDIT_ERR_INVALID_ARG for malformed requests and
 * CREDIT_ERR_NO_LEGAL_PLAN when the shape does not fit.
 */
credit_status_t credit_plan_with(credit_op_t op, int64_t rows, int64_t cols,
                                 credit_dtype_t dtype, int device,
                                 const credit_plan_t *request,
                                 credit_plan_t *out);

/*
 * Row softmax: y[r, j] = exp(x[r, j] - max_r) / sum_k exp(x[r, k] - max_r).
 * (CREDIT "B. Workload-by-Workload Scaling": softmax-logits.)  The partial a
 * CTA pushes is (running max, sum of exp relative to it).
 *   x, y       device, rows x cols of `dtype` (fp32 or bf16); y may equal x
 *   plan       NULL = credit_plan; else a plan from credit_plan[_for] made
 *              for the same op/rows/cols/dtype
 *   workspace  device scratch of >= plan.workspace_bytes (TWO_PASS only;
 *              may be NULL for CLUSTER plans)
 * Fast path: x, y 16-byte aligned and cols*sizeof(dtype) a multiple of 16
 * (bulk copies into shared memory); otherwise an element-wise staging path.
 */
credit_status_t credit_softmax(const void *x, void *y, int64_t rows,
                               int64_t cols, credit_dtype_t dtype,
                               const credit_plan_t *plan, void *workspace,
                               size_t workspace_bytes, void *stream);

/*
 * Row LayerNorm: y = (x - mean) / sqrt(var + eps) * gamma[j] + beta[j], with
 * the biased variance.  (CREDIT "A. Experimental Setup": LayerNorm workload.)
 * The partial a CTA pushes is (count, mean, M2) and the P partials are merged
 * with Chan et al.'s pairwise update in rank order.
 *   gamma, beta  device vectors of `cols` elements of param_dtype, or NULL
 *                (gamma = 1, beta = 0)
 *   eps          >= 0
 * Other arguments as credit_softmax.
 */
credit_status_t credit_layernorm(const void *x, void *y, int64_t rows,
                                 int64_t cols, credit_dtype_t dtype,
                                 const void *gamma, const void *beta,
                                 credit_dtype_t param_dtype, float eps,
                                 const credit_plan_t *plan, void *workspace,
                                 size_t workspace_bytes, void *stream);

/*
 * Row RMSNorm: y = x / sqrt(mean(x^2) + eps) * weight[j].  Not on the CREDIT
 * page; it is the same one-statistic reduce-then-reuse class as LayerNorm.
 * The partial a CTA pushes is its sum of squares.
 *   weight  device vector of `cols` elements of param_dtype, or NULL (= 1)
 * Other arguments as credit_softmax.
 */
credit_status_t credit_rmsnorm(const void *x, void *y, int64_t rows,
                               int64_t cols, credit_dtype_t dtype,
                               const void *weight, credit_dtype_t param_dtype,
                               float eps, const credit_plan_t *plan,
                               void *workspace, size_t workspace_bytes,
                               void *stream);

/*
 * Two-pass call that needs no workspace and allocates no device memory.
 * The CREDIT paper has no counterpart to this entry point; it exists for
 * callers that cannot allocate: programs that gave all device memory to their
 * own pool at start-up, hot loops where cudaMalloc / cudaFree would
 * synchronise the device, plug-in hosts that give the plug-in no allocator.
 * It runs the same two-pass kernels as a CREDIT_TWO_PASS plan, with the
 * per-chunk partials kept in a fixed 2 MiB array inside the library (131072
 * (row, chunk) partials of 16 bytes; every device that loads the library
 * holds the array until the process exits).
 *   op            CREDIT_SOFTMAX, CREDIT_LAYERNORM or CREDIT_RMSNORM
 *   p0, p1        LayerNorm gamma / beta; RMSNorm weight in p0 (p1 ignored);
 *                 softmax ignores both; NULL as in the other entry points
 *   other arguments as credit_layernorm
 * Returns CREDIT_ERR_INVALID_ARG when the call would need more partials than
 * the array holds (rows * ceil(cols / chunk) * 16 bytes > 2 MiB; the chunk
 * is the plan's slice_elems from credit_plan_for(..., CREDIT_TWO_PASS, ...)).
 * The first call on a device looks up the array's device address and sets
 * the kernel attributes of every two-pass kernel this entry point can launch
 * (all three operators, both data and parameter types, aligned and element
 * paths) for that device; make that first call before any stream capture.  All calls share the one array and it keeps the last call's
 * contents (nothing in it needs clearing: every partial is written before it
 * is read); calls whose executions overlap on the GPU, e.g. on two streams,
 * race on it and must be serialised by the caller.
 */
credit_status_t credit_two_pass_noalloc(credit_op_t op, const void *x, void *y,
                                        int64_t rows, int64_t cols,
                                        credit_dtype_t dtype, const void *p0,
                                        const void *p1,
                                        credit_dtype_t param_dtype, float eps,
                                        void *stream);

/* ------------------------------------------------------------------------
 * DSMEM characterisation (CREDIT "C. Positioning": latency, throughput and
 * repeated cluster-synchronisation microbenchmarks with the CTAs on
 * different SMs, median of the runs).  Each benchmark CTA claims more than
 * half of an SM's shared memory, so no two CTAs share an SM; `smids` reports
 * where they ran.  These calls allocate a few bytes of device memory and
 * synchronise the device: they are for calibration, not for a hot path.
 */
typedef enum {
    CREDIT_BENCH_BARRIER = 0,             /* cluster barrier round trip, P CTAs */
    CREDIT_BENCH_EXCHANGE = 1,            /* replicated 16-byte push + barrier, P CTAs */
    CREDIT_BENCH_REMOTE_LOAD_LATENCY = 2, /* pointer chase in a peer's SMEM */
    CREDIT_BENCH_LOCAL_LOAD_LATENCY = 3,  /* the same chase in the CTA's own SMEM */
    CREDIT_BENCH_REMOTE_STORE_BW = 4,     /* one CTA storing 16-byte vectors to a peer */
    CREDIT_BENCH_REMOTE_LOAD_BW = 5,      /* one CTA loading 16-byte vectors from a peer */
    CREDIT_BENCH_LOCAL_STORE_BW = 6,      /* the same stores to its own SMEM */
    CREDIT_BENCH_LOCAL_LOAD_BW = 7,       /* the same loads from its own SMEM */
    CREDIT_BENCH_ASYNC_EXCHANGE = 8       /* st.async 16-byte push to every peer +
                                             wait on the own mbarrier, P CTAs */
} credit_bench_kind_t;

typedef struct {
    int32_t kind;
    int32_t cluster_size;    /* CTAs launched (2 for the pair kinds) */
    int32_t runs;
    int32_t smids[16];       /* SM id of each CTA, rank order (last run) */
    double median_cycles;    /* per operation (barrier, hop, or 64 KiB pass), SM cycles */
    double median_ns;        /* the same in nanoseconds (%globaltimer) */
    double iqr_cycles;       /* interquartile range of the runs, cycles */
    double bytes_per_cycle;  /* throughput kinds: bytes per SM cycle of one CTA */
    double gbps;             /* throughput kinds: GB/s of one CTA */
} credit_bench_result_t;

/*
 * Run one DSMEM microbenchmark on `device`: `iters` operations per launch,
 * `runs` timed launches after one warm-up, median reported.  cluster_size
 * (1..16) applies to the BARRIER, EXCHANGE and ASYNC_EXCHANGE kinds; the
 * other kinds always use a pair of CTAs.  Returns CREDIT_ERR_INVALID_ARG for
 * bad arguments and CREDIT_ERR_DEVICE_TIMEOUT if an exchange wait gave up.
 */
credit_status_t credit_bench_dsmem(int device, int kind, int cluster_size,
                                   int iters, int runs,
                                   credit_bench_result_t *out);

/*
 * Time the work-free control kernel (CREDIT "D. Profitability and Candidate
 * Selection"): `nclusters` clusters of `cluster_size` CTAs of `threads`
 * threads and `smem_bytes` dynamic shared memory, each passing
 * `barriers_per_row` cluster barriers (block barriers when cluster_size is
 * 1) for `rows_per_cluster` rows.  Median over `runs` launches, in
 * microseconds (CUDA events).  T_ctrl of a candidate is its control time
 * minus that of the one-CTA control with the same grid.
 */
credit_status_t credit_control_time(int device, int64_t nclusters,
                                    int cluster_size, int threads,
                                    int64_t smem_bytes, int rows_per_cluster,
                                    int barriers_per_row, int runs,
                                    double *median_us);

/* ------------------------------------------------------------------------
 * Host buffers.  An operator call whose x (and u), y and per-row results live
 * in host memory, pipelined over chunks of rows: library-owned streams carry
 * the host-to-device copies, the kernels and the device-to-host copies, and
 * two device slots alternate between chunks, so the copies in both
 * directions overlap each other and the kernels.  Host buffers should be
 * pinned (cudaHostAlloc) for the copies to overlap; pageable memory works but
 * serialises.  Parameter vectors (p0, p1) are device pointers (they are
 * reused by every chunk).  The call is ordered on `stream` like the other
 * calls: it starts after the stream's earlier work, the stream continues
 * after the last output copy, and nothing waits on the host; the host buffers
 * must stay valid until then.  Concurrent calls on one device share its
 * pipeline streams and run one after the other.
 */
typedef struct {
    credit_op_t op;
    credit_dtype_t dtype;        /* of x, u and y (y is int8 for quantization) */
    int64_t rows, cols;
    const void *x;               /* host, rows x cols */
    const void *u;               /* host, Pearson's second operand, else NULL */
    void *y;                     /* host, rows x cols */
    float *row_out;              /* host, per-row scales (quantization) or r
                                    (Pearson), rows floats, else NULL */
    const void *p0, *p1;         /* device gamma/beta, weight or weights, may be NULL */
    credit_dtype_t param_dtype;
    float eps;
} credit_host_call_t;

/* Device bytes credit_run_host needs for `rows_per_chunk`-row chunks (two
 * slots of inputs and outputs, plus the two-pass workspace if `plan` is a
 * TWO_PASS plan).  No CUDA call. */
credit_status_t credit_host_buffer_bytes(const credit_host_call_t *call,
                                         const credit_plan_t *plan,
                                         int64_t rows_per_chunk, size_t *bytes);

/* Run `call` over chunks of rows_per_chunk rows (the last may be shorter)
 * with `plan` (not NULL; e.g. credit_plan or credit_plan_profiled for the
 * chunk's shape -- each chunk re-derives it for its row count), using the
 * caller's 256-byte-aligned device_buffer of at least
 * credit_host_buffer_bytes bytes.  Returns CREDIT_ERR_INVALID_ARG for missing
 * pointers or a short buffer; otherwise the status of the first failing
 * chunk, if any. */
credit_status_t credit_run_host(const credit_host_call_t *call,
                                const credit_plan_t *plan, void *device_buffer,
                                size_t device_buffer_bytes,
                                int64_t rows_per_chunk, void *stream);

/* ------------------------------------------------------------------------
 * Profitability cost model (CREDIT "D. Profitability and Candidate
 * Selection").  For one shape it times the non-DSMEM baseline -- the fastest
 * of the one-CTA-per-row local-staging kernel (when a row fits one CTA's
 * shared memory), the warp-per-row register kernel (rows of at most 4 KiB)
 * and the two-pass global re-read pair -- and predicts every legal clustered
 * candidate (each P with its whole slice staged, where it fits, and with the
 * L2-tail plans sized for two, three and -- where the four-CTA instantiation
 * exists -- four CTAs per SM, and with half the three-CTA staged length) from
 * measured primitives, without timing the candidate:
 *     T(P) = B_credit / (R_loc(c_eff, f) * S(P)) * q + T_ctrl(P) + T_comm(P)
 *            + T_replay(P)
 *   R_loc(c, f)  the local-work primitive: the one-CTA-per-row kernel (no
 *                DSMEM) timed once per operator and dtype on calibration
 *                rows that let c = 1..8 CTAs share an SM, fully staged and
 *                with a half and three quarters of each row an L2 tail (the
 *                tail levels also at residencies only tail plans reach);
 *                piecewise linear in c and in the tail fraction f
 *   c_eff        the CTAs per SM the candidate keeps resident: resident
 *                clusters x P / SMs, at most what its footprint allows (a
 *                cluster lives in one GPC, so clusters may not fill every slot)
 *   S(P)         the synchronisation factor of cluster size P: the clustered
 *                kernel timed once per operator on calibration rows of P
 *                slices (three CTAs per SM), over R_loc at the residency it
 *                reached -- what waiting for a cluster's slowest CTA costs
 *   q            the last wave's fill: ceil(rows / clusters) clusters / rows
 *   T_ctrl(P)    the work-free control kernel with the candidate's grid,
 *                cluster size, footprint and two barriers per row, minus the
 *                same grid without clusters
 *   T_comm(P)    waves x the measured exchange's cost beyond one cluster
 *                barrier (DSMEM profile: the st.async exchange for ASYNC plans,
 *                push + barrier for BARRIER plans, clamped at zero)
 *   T_replay(P)  waves x P shared-memory reads: every CTA folds the P partials
 *                locally (DSMEM profile: one local load hop)
 * The deposit residual [T_wSMEM - T_input]+ is zero: a 16-byte push per peer
 * is far below the per-SM input stream.  The candidate with the smallest
 * prediction is kept if it beats T_base, else the baseline.  As on the
 * pages, the model screens and a final tuning step may pick another legal
 * size: with tune > 0 the `tune` best-predicted cluster sizes are timed (all
 * their staging forms, and the persistent and pipelined kernels of the same
 * P); the three fastest are timed twice more, interleaved, and the plan with
 * the smallest mean of its three medians is chosen if it beats the baseline.
 */
typedef struct {
    int32_t cluster_size;    /* P; 1 = the baseline */
    int32_t legal;           /* 0: the slice does not fit / no residency */
    credit_plan_t plan;
    double t_ctrl_us;        /* control time excess over the baseline's control */
    double t_comm_us;        /* push cost beyond the barrier, all waves */
    double pred_us;          /* predicted time */
    double measured_us;      /* tuning: measured time of `plan` (0 = not timed) */
    double persistent_us;    /* tuning: measured time of the persistent kernel
                                of this P (0 = not timed or not legal) */
    double pipelined_us;     /* tuning: measured time of the warp-specialised
                                persistent kernel of this P (0 = not timed or
                                not legal) */
    double tail_us;          /* tuning: measured time of the fastest L2-tail
                                plan of this P (0 = none timed) */
    int64_t tail_staged_elems;  /* that plan's staged_elems */
} credit_candidate_t;

typedef struct {
    int32_t baseline_variant;     /* CREDIT_CLUSTER (P = 1 staging), CREDIT_WARP_ROWS
                                     or CREDIT_TWO_PASS */
    int32_t model_cluster_size;   /* the model's pick (1 = the baseline) */
    int32_t profitable;           /* 1 if a clustered candidate is predicted faster */
    int32_t chosen_cluster_size;  /* after tuning (equals the model's pick if tune = 0) */
    int32_t chosen_variant;       /* variant of the chosen plan */
    int32_t reserved;
    double t_base_us;             /* measured baseline time (median) */
    double b_base_bytes;          /* bytes the baseline moves */
    double b_credit_bytes;        /* bytes a clustered candidate moves */
    double t_ctrl_base_us;        /* the baseline's control time */
    credit_candidate_t cand[16];  /* index P - 1; [0] describes the baseline */
} credit_model_report_t;

/*
 * Run the DSMEM microbenchmarks the cost model uses (cluster barrier,
 * replicated push and st.async exchange for P = 2..16, median of `runs`) on
 * `device` and keep the profile in memory.  If profile_path is not NULL the
 * profile is also written there as JSON.  Synchronises the device; allocates
 * a few bytes.
 */
credit_status_t credit_calibrate(int device, int runs, const char *profile_path);

/*
 * The persisted calibration profile.  A profile file holds the DSMEM profile
 * of credit_calibrate and the plans credit_plan_profiled chose per shape, so
 * a later process plans without recalibrating or re-timing candidates.  It
 * is keyed on what produced it: the device key below and the library
 * version; a profile whose key differs from the loading device's is stale.
 * Nothing on the CREDIT pages corresponds to this; the pages recalibrate per
 * run.
 *
 * Environment (read by the library):
 *   CREDIT_PROFILE=<path>  the first planning call on a device loads <path>
 *                          when it exists and is not stale; every calibration
 *                          and profiled plan then writes the device's state
 *                          back to <path> (atomically: a temporary file
 *                          renamed over it)
 *   CREDIT_FORCE=<plan>    automatic plans become <plan> where it is legal
 *                          for the shape (else the automatic choice stands):
 *                          cluster:P, cluster:PxR (R rows per cluster),
 *                          cluster:P:sN (an L2-tail plan staging N elements),
 *                          cluster:P:sN:tT (the same with T threads per CTA),
 *                          persist:P, pipe:P, warp_rows or twopass
 */
typedef struct {
    char gpu_name[96];
    int32_t sms;
    int32_t sm_clock_mhz;    /* peak SM clock */
    int32_t mem_clock_mhz;   /* peak memory clock */
    int32_t cc_major;
    int32_t cc_minor;
    int32_t reserved;
} credit_device_key_t;

/* The key of `device` (host query).  CREDIT_ERR_CUDA if it cannot be read. */
credit_status_t credit_device_key(int device, credit_device_key_t *out);

/* Write the DSMEM profile (if calibrated) and every chosen plan of `device`
 * to `path`.  CREDIT_ERR_INVALID_ARG if the file cannot be written. */
credit_status_t credit_save_profile(int device, const char *path);

/* Load `path` into `device`'s in-memory state: its DSMEM profile and its
 * chosen plans (each re-derived on this device; one it cannot launch is
 * skipped).  Returns CREDIT_ERR_INVALID_ARG for a missing, unreadable or
 * malformed file and CREDIT_ERR_NOT_CALIBRATED, loading nothing, for a
 * stale profile (another GPU, SM count, clock, compute capability or
 * library version). */
credit_status_t credit_load_profile(int device, const char *path);

/* Host-only check of a profile file against a device key: CREDIT_OK if it
 * matches `key` and this library version, CREDIT_ERR_NOT_CALIBRATED if it is
 * stale, CREDIT_ERR_INVALID_ARG if it is not a readable profile. */
credit_status_t credit_profile_check(const char *path, const credit_device_key_t *key);

/*
 * The staged-copy primitive: every CTA moves one footprint of bytes from HBM
 * into its shared memory (non-multicast bulk copies, an mbarrier per 16 KiB),
 * folds it once as the chunks land, meets at a block barrier, and reads it
 * again to store it back to HBM with streaming stores -- a one-pass
 * reduce-reuse CTA's data movement and shared-memory passes without its
 * arithmetic or exchange.  The footprint is the largest multiple of
 * 16 KiB that lets `ctas_per_sm` (1..8) CTAs share an SM, the grid moves at
 * least 512 MiB, and *gbps is (bytes read + written) / median time of `runs`
 * launches (CUDA events).  *resident (may be NULL) receives the CTAs per SM
 * the occupancy calculator reports for that footprint.  Allocates and frees
 * the buffers; synchronises the device.
 */
credit_status_t credit_stage_copy_rate(int device, int ctas_per_sm, int runs,
                                       double *gbps, int *resident);

/*
 * The L2 read primitive: every resident CTA (512 threads, as many per SM as
 * fit) reads a whole window of window_bytes (64 KiB .. 64 MiB, a multiple of
 * 16) with 16-byte loads that bypass L1, eight in flight per thread.  The
 * window lies well inside the L2, so every read after the warm-up launch hits,
 * so *gbps = (CTAs x window bytes) / median time of `runs` launches is the
 * rate at which the SMs can pull data from L2 -- the ceiling of an operator
 * whose per-column parameters are re-read from L2 for every row (CREDIT "D.
 * Traffic Validation" counts only DRAM bytes; this is the on-chip side).
 * Allocates and frees the window; synchronises the device.
 */
credit_status_t credit_l2_read_rate(int device, int64_t window_bytes, int runs,
                                    double *gbps);

/*
 * Apply the cost model to one shape on `device` (calibrating first if
 * needed).  Allocates scratch x / y / parameter / workspace buffers for the
 * shape's first rows -- all of them up to 1 GiB of input, fewer beyond --
 * filled with hashed values, times the baseline (median of `runs`), runs the
 * control kernels, fills `report` (may be NULL; its times are those of the
 * timed rows) and writes the chosen plan, planned for every row, to `out`.  param_dtype is the parameters' dtype, or -1 for none; tune is the
 * number of best-predicted candidates to time (0 = the model alone).  The choice
 * is cached: later credit_plan calls for the same (op, rows, cols, dtype,
 * device) return it.  Synchronises the device.
 */
credit_status_t credit_plan_profiled(credit_op_t op, int64_t rows,
                                     int64_t cols, credit_dtype_t dtype,
                                     int param_dtype, int device, int runs,
                                     int tune, credit_plan_t *out,
                                     credit_model_report_t *report);

/*
 * Row-wise symmetric int8 quantization (CREDIT "B. Workload-by-Workload
 * Scaling" and "D. Traffic Validation": the quantization workload, a 4-byte
 * read and a 1-byte write per element for fp32 input).  Per row:
 *   amax = max |x_j|,  scale = amax / 127 (fp32),
 *   q_j = clamp(round_half_even(x_j / scale), -127, 127)  (IEEE fp32 division)
 * and q = 0, scale = 0 for an all-zero row.  The partial a CTA pushes is its
 * absmax.
 *   x       device, rows x cols of `dtype` (fp32 or bf16)
 *   q       device, rows x cols int8 codes; must not overlap x or scales
 *   scales  device, rows fp32 scales (4-byte aligned)
 * The bulk path also needs cols to be a multiple of 16.  Persistent plans are
 * not offered for this operator.  Other arguments as credit_softmax.
 */
credit_status_t credit_quantize(const void *x, int8_t *q, float *scales,
                                int64_t rows, int64_t cols,
                                credit_dtype_t dtype,
                                const credit_plan_t *plan, void *workspace,
                                size_t workspace_bytes, void *stream);

/*
 * Row-wise weighted standardization (the weighted-variance workload of
 * CREDIT "B. Workload-by-Workload Scaling", read as the weighted counterpart
 * of LayerNorm): with per-column weights w_j >= 0,
 *   W = sum w_j,  mean = sum w_j x_j / W,  var = sum w_j (x_j - mean)^2 / W,
 *   y_j = (x_j - mean) / sqrt(var + eps).
 * The partial a CTA pushes is (W_q, mean_q, M2_q), merged like LayerNorm's with
 * weight sums in place of counts.  Rows whose weights sum to 0 produce
 * unspecified values.
 *   weights       device vector of cols weights of weight_dtype (not NULL)
 * Persistent plans are not offered for this operator.  Other arguments as
 * credit_layernorm.
 */
credit_status_t credit_weighted_std(const void *x, void *y, int64_t rows,
                                    int64_t cols, credit_dtype_t dtype,
                                    const void *weights,
                                    credit_dtype_t weight_dtype, float eps,
                                    const credit_plan_t *plan, void *workspace,
                                    size_t workspace_bytes, void *stream);

/*
 * Row-wise Pearson correlation of two matrices x and u of the same shape
 * (the Pearson workload of CREDIT "B. Workload-by-Workload Scaling"; the
 * pages name it only, and this reading keeps the reduce-then-reuse shape):
 *   mx, mu    row means;  vx, vu  biased variances;  cxu  covariance,
 *   y_j = (x_j - mx)(u_j - mu) / (sqrt(vx + eps) sqrt(vu + eps)),
 *   r   = cxu / (sqrt(vx + eps) sqrt(vu + eps))      (Pearson's r at eps = 0),
 * so the row mean of y is r.  Each CTA stages its slice of both operands
 * (so P is twice that of a one-operand row) and pushes (n, mx, mu) and
 * (Mxx, Muu, Cxu) -- two 16-byte slots -- to every peer; co-moments merge
 * in the parallel-axis form of Chan et al.
 *   x, u      device inputs, rows x cols, dtype (u not NULL)
 *   y         device output like x; may equal x or u (in place), may not
 *             partially overlap either
 *   r         device output, rows fp32 correlations, 4-byte aligned, not
 *             overlapping x, u or y
 *   eps       >= 0; a row with a constant operand and eps = 0 gives
 *             unspecified values
 * Persistent plans and rows_per_cluster > 1 are not offered for this
 * operator; TWO_PASS needs rows * ceil(cols / chunk) * 32 bytes of
 * workspace (plan.workspace_bytes).  Other arguments as credit_softmax.
 */
credit_status_t credit_pearson(const void *x, const void *u, void *y, float *r,
                               int64_t rows, int64_t cols, credit_dtype_t dtype,
                               float eps, const credit_plan_t *plan,
                               void *workspace, size_t workspace_bytes,
                               void *stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char *credit_status_string(credit_status_t status);

/*
 * Read and clear the device error word of `device`.  Bounded device waits
 * that give up set it (CREDIT_ERR_DEVICE_TIMEOUT), and so do the index checks
 * of the checked build (CREDIT_ERR_DEVICE_BOUNDS; a timeout is reported
 * first when both happened); CREDIT_OK otherwise.  Synchronises the device.
 */
credit_status_t credit_get_device_error(int device);

/*
 * Exercise the bounded-wait path on `device`: a one-thread kernel waits on an
 * mbarrier that nothing completes, gives up after limit_ns (1 us .. 1 s) and
 * sets the device error word, which is then read and cleared.  Returns
 * CREDIT_ERR_DEVICE_TIMEOUT when the path works.  The kernel ends by itself
 * (no copy in flight, no cluster barrier), so the context stays usable.
 */
credit_status_t credit_selftest_wait_timeout(int device, int64_t limit_ns);

/*
 * The checked build (libcredit_checked.so, compiled with -DCREDIT_DEBUG) runs
 * the same kernels with index checks on the staged-slice, ring-slot, chunk
 * mbarrier and exchange-slot accesses: a failed check records
 * CREDIT_ERR_DEVICE_BOUNDS in the device error word and skips the access
 * instead of touching memory outside the buffer.  It also records a phase
 * trace of the one-row-per-cluster kernel (below).  The regular build has
 * neither.
 *
 * credit_debug_build: 1 for the checked build, 0 otherwise.
 */
int credit_debug_build(void);

/*
 * Exercise the index-check path on `device`: a one-thread kernel records a
 * failed check (no memory outside any buffer is touched) and the device error
 * word is read and cleared.  Returns CREDIT_ERR_DEVICE_BOUNDS in the checked
 * build, CREDIT_ERR_UNSUPPORTED in the regular one.
 */
credit_status_t credit_selftest_bounds(int device);

/*
 * Phase trace of the last launches of the one-row-per-cluster kernel on the
 * current device (checked build only).  Each CTA with blockIdx.x <
 * CREDIT_TRACE_CTAS records, from thread 0, 8 unsigned 64-bit words: the
 * %globaltimer (ns) at kernel entry, after its bulk copies are issued, after
 * its statistics are folded, after the CTA partial, after the exchange and
 * combine, after its output, at exit, and its SM id.  Stamps of a CTA index
 * are overwritten by every launch that reaches it.  Copies `ctas` * 64 bytes
 * (ctas <= CREDIT_TRACE_CTAS) into `host`; CREDIT_ERR_UNSUPPORTED in the
 * regular build.  Synchronises the device.
 */
#define CREDIT_TRACE_CTAS 8192
credit_status_t credit_debug_trace(void *host, int64_t ctas);

/*
 * Combined statistics every CTA rebuilt (checked build only).  The protocol's
 * all-gather rests on each of a cluster's P CTAs reconstructing the full row
 * statistic on its own from the same P partials in the same rank order
 * (CREDIT "C. Cluster Reduction and Reuse Protocol", All-Gather Trade-off and
 * Output Generation), so every CTA must hold bit-identical values.  The
 * clustered, persistent, warp-specialised and Pearson kernels record, for
 * rows r < CREDIT_DEBUG_STATS_ROWS of a launch, from thread 0 of CTA `rank`,
 * 8 floats at host[(r * 16 + rank) * 8]: the statistics (softmax m, s;
 * LayerNorm / weighted standardization n, mean, M2; RMSNorm sum of squares;
 * quantization absmax; Pearson n, mean x, mean u, Mxx, Muu, Cxu), unused
 * slots, and the cluster size P in the last.  Copies `rows` (<=
 * CREDIT_DEBUG_STATS_ROWS) rows of 16 records into `host`, then resets the
 * record to all-ones bytes (NaN), so entries no CTA wrote read as NaN.
 * CREDIT_ERR_UNSUPPORTED in the regular build.  Synchronises the device.
 */
#define CREDIT_DEBUG_STATS_ROWS 64
credit_status_t credit_debug_stats(void *host, int64_t rows);

/* Library version as "major.minor.patch" (static storage). */
const char *credit_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CREDIT_H */
