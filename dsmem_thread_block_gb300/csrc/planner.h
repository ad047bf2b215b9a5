// planner.h -- device facts, per-kernel facts and the plan builders.
#pragma once

#include <cstdint>

#include "credit.h"

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
credit_status_t make_plan(int dev, credit_op_t op, int64_t rows, int64_t cols,
                          credit_dtype_t dtype, credit_variant_t variant, int P,
                          int threads, int cps, credit_plan_t* out, int64_t chunk = 0,
                          int rows_per_cluster = 0);

// Bytes between the staged row slices of a multi-row CTA.
int64_t row_pitch(int64_t slice_elems, int elem_bytes);

// The plan the profiled cost model chose for this shape, if it has run.
bool lookup_profiled_plan(int dev, credit_op_t op, int64_t rows, int64_t cols,
                          credit_dtype_t dtype, credit_plan_t* out);

// The automatic plan: the profiled choice when there is one, else a static
// rule.
credit_status_t auto_plan(int dev, credit_op_t op, int64_t rows, int64_t cols,
                          credit_dtype_t dtype, credit_plan_t* out);

}  // namespace credit
