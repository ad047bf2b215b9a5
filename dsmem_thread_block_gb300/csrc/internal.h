// internal.h -- declarations shared between the host API (api.cu) and the
// translation units that own the kernels.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

namespace credit {

// Arguments of the clustered reduce-reuse kernel (one launch = all rows).
struct ClusterArgs {
    const void* x;
    void* y;
    const void* p0;       // gamma (LayerNorm), weight (RMSNorm, weighted std) or u (Pearson)
    const void* p1;       // beta (LayerNorm), may be null
    int64_t rows;         // rows of this launch (the last cluster may hold fewer than R)
    int64_t cols;
    int64_t slice;        // elements owned by one CTA (multiple of the vector width)
    int32_t chunk_elems;  // elements per bulk copy / mbarrier
    int32_t pitch;        // bytes between the staged slices of a CTA's rows
    float eps;
    unsigned* err;        // device error word
    float* aux;           // per-row scales (quantization) or r (Pearson) out
    int32_t exchange;     // 0: push + cluster barrier; 1: st.async deposits + mbarrier
    float* dbg_stats;     // checked build: per-(row, rank) combined statistics out (or null)
    int64_t staged;       // elements of a CTA's slice staged in shared memory (>= slice: all);
                          // the rest, the L2 tail, is read twice through L2
};

constexpr int kMaxRowsPerCluster = 4;

// Operators and data types whose one-row-per-cluster kernel can leave an L2
// tail of its slice unstaged (not fp32 softmax, whose stash pass rewrites
// the staged slice in place).
__host__ __device__ constexpr bool tail_capable(int op, int dtype_bytes) {
    return op == 1 /* LayerNorm */ || op == 2 /* RMSNorm */ || (op == 0 && dtype_bytes == 2);
}

// Operators and data / parameter types with a one-row-per-cluster
// instantiation bounded to 64 registers, four CTAs per SM, for L2-tail plans
// whose footprint leaves room for four: bf16 softmax and LayerNorm with bf16
// data and fp32 parameters (no spills at that bound; both measured faster).
// RMSNorm's pipelined weight loads spill there and measured slower.
__host__ __device__ constexpr bool quad_capable(int op, int dtype_bytes, int param_bytes) {
    return dtype_bytes == 2 &&
           (op == 0 /* softmax */ || (op == 1 /* LayerNorm */ && param_bytes == 4));
}

// Arguments of the two-pass (global re-read) kernel pair.
struct TwoPassArgs {
    const void* x;
    void* y;
    const void* p0;
    const void* p1;
    int64_t cols;
    int32_t chunk;        // elements per block (threads * kTwoPassVpt * vector)
    int32_t nch;          // chunks per row
    float eps;
    float* ws;            // rows * nch * 4 floats (8 for Pearson)
    float* aux;           // per-row scales (quantization) or r (Pearson) out
};

constexpr int kTwoPassVpt = 4;  // 16-byte vectors per thread per chunk

// Arguments of the persistent clustered kernel: `nclusters` resident clusters
// loop over the rows; each CTA streams its slice of every row it owns through
// a ring of `nslots` shared-memory slots of `chunk` elements.
struct PersistArgs {
    const void* x;
    void* y;
    const void* p0;
    const void* p1;
    int64_t rows;
    int64_t cols;
    int32_t slice;        // elements owned by one CTA (multiple of the vector width)
    int32_t chunk;        // elements per ring slot / bulk copy (multiple of the vector width)
    int32_t nslots;       // ring slots per CTA (<= kPersistMaxSlots)
    int32_t nclusters;    // clusters in the grid
    float eps;
    unsigned* err;
    int32_t exchange;     // 0: push + cluster barrier per row; 1: st.async deposits + mbarrier
    int32_t reducers;     // 0: one consumer role; > 0: reducer warps of the warp-specialised kernel
    int32_t param_off;    // warp-specialised kernel: byte offset of the parameter room in
                          // dynamic shared memory (0 = none)
    int32_t param_room;   // bytes of that room
    float* dbg_stats;     // checked build: per-(row, rank) combined statistics out (or null)
};

constexpr int kPersistMaxSlots = 32;
constexpr int kPersistMaxThreads = 544;  // 16 consumer warps + 1 producer warp

// Arguments of the warp-per-row kernel (rows that fit one warp's registers).
struct WarpRowsArgs {
    const void* x;
    void* y;
    const void* p0;
    const void* p1;
    int64_t rows;
    int64_t cols;
    float eps;
};

constexpr int kWarpRowNV = 8;          // 16-byte vectors per lane: rows up to 4 KiB
constexpr int kWarpRowThreads = 256;

// Kernel selector: op 0..2, dtype 0 = fp32 / 1 = bf16, pdtype likewise,
// vec = aligned 16-byte path, rows = rows per cluster (1, 2 or 4; the
// element path has 1).
struct KernelKey {
    int op, dtype, pdtype;
    bool vec;
    int rows = 1;
    bool deep = false;  // clustered kernel for slices that leave room for <= 2 CTAs per SM
    bool quad = false;  // clustered kernel bounded to 64 registers: four CTAs per SM
};

const void* cluster_kernel(KernelKey k);
// Pearson correlation (two staged operands): dtype 0 = fp32 / 1 = bf16
const void* pearson_cluster_kernel(int dtype, bool vec);
const void* pearson_stats_kernel(int dtype, bool vec);
const void* pearson_apply_kernel(int dtype, bool vec);
const void* persistent_kernel(KernelKey k);
const void* pipelined_kernel(KernelKey k);  // warp-specialised persistent form
// Reducer warps of the warp-specialised kernel for `consumer_warps` consumer warps.
int pipelined_reducers(int op, int dtype, int consumer_warps);
const void* two_pass_stats_kernel(KernelKey k);
// the instantiation for rows of `nvec` 16-byte vectors (null when none fits)
const void* warp_rows_kernel(KernelKey k, int64_t nvec);
const void* two_pass_apply_kernel(KernelKey k);

cudaError_t launch_cluster(KernelKey k, const ClusterArgs& a, int P, int threads, size_t smem,
                           cudaStream_t s);
cudaError_t launch_persistent(KernelKey k, const PersistArgs& a, int P, int threads,
                              size_t smem, cudaStream_t s);
cudaError_t launch_two_pass(KernelKey k, const TwoPassArgs& a, int64_t rows,
                            int threads, cudaStream_t s);
cudaError_t launch_warp_rows(KernelKey k, const WarpRowsArgs& a, int blocks, cudaStream_t s);

unsigned* device_error_word();  // address of this device's error word
// checked build: this device's per-(row, rank) statistics record (null in the
// regular build)
float* debug_stats_buffer();

}  // namespace credit
