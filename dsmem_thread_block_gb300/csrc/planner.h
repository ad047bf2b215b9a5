// planner.h -- device facts, per-kernel facts and the plan builders.
#pragma once

#include <cstdint>
#include <vector>

#include "credit.h"
#include "internal.h"

namespace credit {

constexpr int kMaxDevices = 64;

struct DevInfo {
    bool valid = false;
    int sms = 0;
    int smem_optin = 0;      // max dynamic + static shared memory per block
    int smem_per_sm = 0;
    int reserved_smem = 0;   // shared memory the system reserves per block
    int l2_bytes = 0;
    int major = 0, minor = 0;
    int max_threads_sm = 0;
    int regs_per_sm = 0;
};

struct KernelInfo {
    int static_smem = 0;
    int max_dyn_smem = 0;
    int regs = 0;
};

const DevInfo* device_info(int dev);
const KernelInfo* kernel_info(int dev, const void* fn, bool cluster);
int occupancy_clusters(int dev, const void* fn, int P, int threads, size_t smem, int64_t rows);

// Elements per bulk copy (one mbarrier each) for a staged slice of a CTA
// that stages `rows_per_cluster` rows.
int64_t bulk_chunk_elems(int64_t slice_elems, int elem_bytes, int rows_per_cluster);

// Build the plan of a given variant (threads == 0 / cps == 0 / chunk == 0:
// choose).  cps is the number of persistent CTAs meant to share one SM (1 or
// 2); chunk the persistent ring's slot size in elements (a power-of-two
// number of 16-byte vectors).
// staged: CREDIT_CLUSTER with one row per cluster, the elements of each
// CTA's slice to stage in shared memory (0 = all); the rest is an L2 tail.
credit_status_t make_plan(int dev, credit_op_t op, int64_t rows, int64_t cols,
                          credit_dtype_t dtype, credit_variant_t variant, int P,
                          int threads, int cps, credit_plan_t* out, int64_t chunk = 0,
                          int rows_per_cluster = 0, int64_t staged = 0);

// Dynamic shared memory of one CTA of an L2-tail plan that `cps` CTAs can
// share an SM with: whole kilobytes, the kernel's static shared memory
// rounded up to one, and a kilobyte of slack.
int64_t tail_budget_bytes(const DevInfo& d, int static_smem, int cps);

// Does a one-row-per-cluster launch of `smem_bytes` dynamic shared memory
// leave room for fewer than three CTAs per SM?  Then it takes the deep
// instantiation (where the operator has one), whose launch bounds allow two
// CTAs per SM and twice the registers.
bool deep_footprint(int dev, KernelKey k, int64_t smem_bytes);

// Does a one-row-per-cluster L2-tail launch (`tail`) of `smem_bytes` dynamic
// shared memory leave room for four CTAs per SM, for an operator with the
// four-CTA instantiation?  Then it takes that instantiation.
bool quad_footprint(int dev, KernelKey k, int64_t smem_bytes, bool tail);

// Columns of one CTA's slice of a row split over P CTAs of the
// one-row-per-cluster kernel: whole 128-byte lines, so that no two CTAs share
// a line of the row and each slice's bulk copies start on a line boundary
// (when the row does).  The last CTA takes the remainder; trailing CTAs may
// be empty.
int64_t cluster_slice(int64_t cols, int P, int es);

// Staged elements per row of an L2-tail plan of cluster size P with
// rows_per_cluster rows per cluster that lets `cps` CTAs share an SM, or 0
// when the operator has no L2-tail form or the whole slice already fits.
int64_t tail_staged_for(int dev, credit_op_t op, int64_t cols, credit_dtype_t dtype, int P,
                        int cps, int rows_per_cluster = 1);

// Bytes between the staged row slices of a multi-row CTA.
int64_t row_pitch(int64_t slice_elems, int elem_bytes);

// The plan the profiled cost model chose for this shape, if it has run.
bool lookup_profiled_plan(int dev, credit_op_t op, int64_t rows, int64_t cols,
                          credit_dtype_t dtype, credit_plan_t* out);

// Calibration-profile state of the cost model (costmodel.cu) and its
// persistence (profile.cu).
struct ChosenPlan {
    int op, dtype;
    int64_t rows, cols;
    credit_plan_t plan;
};
// The DSMEM profile: per cluster size (index P, 17 entries) the cluster
// barrier, the replicated push + barrier exchange and the st.async exchange;
// and the local replay cost, one hop of a shared-memory pointer chase.
constexpr int kProfileSizes = 17;
struct DsmemData {
    double barrier_ns[kProfileSizes];
    double exchange_ns[kProfileSizes];
    double async_ns[kProfileSizes];
    double local_load_ns;
};
bool dsmem_profile_get(int dev, DsmemData* out);
void dsmem_profile_set(int dev, const DsmemData& d);
// The local-work primitive of one (operator, dtype, parameter dtype): GB/s
// (one read and one write of the matrix) of the one-CTA-per-row kernel at
// 1..kLocalMaxCps CTAs per SM ([0] unused), fully staged and with an L2 tail
// of a half and of three quarters of each row (0 where the operator has no
// L2-tail form or the residency cannot be reached).
// sync[P] (P = 2..16) is the clustered kernel's synchronisation factor: its
// rate at cluster size P on calibration rows that give three CTAs per SM
// over the local rate at the same effective residency (1 = no cost; 0 =
// not measured).
constexpr int kLocalMaxCps = 8;
struct LocalRates {
    int op, dtype, pdt;
    double full[kLocalMaxCps + 1];
    double tail50[kLocalMaxCps + 1];
    double tail75[kLocalMaxCps + 1];
    double sync[kProfileSizes];
};
std::vector<LocalRates> local_rates(int dev);
void local_rates_put(int dev, const LocalRates& r);
std::vector<ChosenPlan> chosen_plans(int dev);
void chosen_plan_put(int dev, const ChosenPlan& c);
// CREDIT_PROFILE: load the named profile once per device (if it exists and
// matches this device and library), and save the state back after a
// calibration or a profiled plan.  No-ops when the variable is unset.
void profile_env_load(int dev);
void profile_env_save(int dev);
// CREDIT_FORCE: the plan it names for this shape, if set and legal.
bool forced_plan(int dev, credit_op_t op, int64_t rows, int64_t cols, credit_dtype_t dtype,
                 credit_plan_t* out);

// The automatic plan: the profiled choice when there is one, else a static
// rule.
credit_status_t auto_plan(int dev, credit_op_t op, int64_t rows, int64_t cols,
                          credit_dtype_t dtype, credit_plan_t* out);

}  // namespace credit
