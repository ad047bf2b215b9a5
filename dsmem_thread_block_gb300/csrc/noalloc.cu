// noalloc.cu -- a two-pass entry point that needs no workspace from the
// caller and allocates no device memory.
//
// The two-pass baseline keeps one 16-byte partial per (row, chunk) between
// its two kernels.  Normally the caller passes that workspace in.  Some
// callers cannot hand one over: code that gave all of the device's memory to
// its own pool at start-up (a cudaMalloc there fails or fragments the pool),
// hot loops where a cudaMalloc / cudaFree would synchronise the whole device,
// and plug-in hosts that expose no allocator to the plug-in.  For them the
// partials live in a fixed array inside the library instead.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "credit.h"
#include "common.cuh"
#include "internal.h"
#include "planner.h"

namespace credit {
namespace {

// 2 MiB of partials: 131072 (row, chunk) pairs.  Every device that loads the
// library holds this array until the process exits.
constexpr size_t kStaticScratchBytes = size_t(2) << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices];  // device address of g_static_scratch, per device

// Per-device set-up, once per device with `dev` current: the device address
// of the array (in host code `g_static_scratch` names a host-side shadow, not
// device memory, so the address has to come from the runtime) and the kernel
// attributes of every two-pass kernel this entry point can launch for `op`
// (both data types, aligned and element paths, both parameter types), so
// that no later call does lazy per-device work.
void* scratch_address(int dev) {
    std::lock_guard<std::mutex> lk(g_setup_mu);
    if (!g_scratch_addr[dev]) {
        for (int op : {(int)kSoftmax, (int)kLayerNorm, (int)kRMSNorm}) {
            for (int dt = 0; dt < 2; ++dt) {
                for (int pdt = 0; pdt < 2; ++pdt) {
                    for (bool vec : {true, false}) {
                        const KernelKey k{op, dt, pdt, vec};
                        const void* fs = two_pass_stats_kernel(k);
                        const void* fa = two_pass_apply_kernel(k);
                        if ((fs && !kernel_info(dev, fs, false)) ||
                            (fa && !kernel_info(dev, fa, false)))
                            return nullptr;
                    }
                }
            }
        }
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

}  // namespace
}  // namespace credit

using namespace credit;

extern "C" credit_status_t credit_two_pass_noalloc(credit_op_t op, const void* x, void* y,
                                                   int64_t rows, int64_t cols,
                                                   credit_dtype_t dtype, const void* p0,
                                                   const void* p1, credit_dtype_t param_dtype,
                                                   float eps, void* stream) {
    if (!x || !y || rows < 1 || cols < 1) return CREDIT_ERR_INVALID_ARG;
    if (op != CREDIT_SOFTMAX && op != CREDIT_LAYERNORM && op != CREDIT_RMSNORM)
        return CREDIT_ERR_UNSUPPORTED;
    if (dtype != CREDIT_F32 && dtype != CREDIT_BF16) return CREDIT_ERR_UNSUPPORTED;
    if (op == CREDIT_SOFTMAX) p0 = p1 = nullptr;
    if (op == CREDIT_RMSNORM) p1 = nullptr;
    if ((p0 || p1) && param_dtype != CREDIT_F32 && param_dtype != CREDIT_BF16)
        return CREDIT_ERR_UNSUPPORTED;
    if (op != CREDIT_SOFTMAX && !(eps >= 0.f)) return CREDIT_ERR_INVALID_ARG;
    const int64_t es = dtype == CREDIT_F32 ? 4 : 2;
    if (rows > INT64_MAX / cols || rows * cols > INT64_MAX / es) return CREDIT_ERR_INVALID_ARG;
    const uintptr_t xb = (uintptr_t)x, yb = (uintptr_t)y, bytes = (uintptr_t)(rows * cols * es);
    if (xb != yb && xb < yb + bytes && yb < xb + bytes) return CREDIT_ERR_INVALID_ARG;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return CREDIT_ERR_CUDA; }
    if (dev < 0 || dev >= kMaxDevices) return CREDIT_ERR_CUDA;
    credit_plan_t plan;
    const credit_status_t st =
        make_plan(dev, op, rows, cols, dtype, CREDIT_TWO_PASS, 0, 0, 0, &plan);
    if (st != CREDIT_OK) return st;
    if ((size_t)plan.workspace_bytes > kStaticScratchBytes) return CREDIT_ERR_INVALID_ARG;
    void* scratch = scratch_address(dev);
    if (!scratch) return CREDIT_ERR_CUDA;

    const auto a16 = [](const void* p) { return ((uintptr_t)p & 15u) == 0; };
    const bool vec = a16(x) && a16(y) && (cols * es) % 16 == 0 && (!p0 || a16(p0)) &&
                     (!p1 || a16(p1));
    const KernelKey key{(int)op, (int)dtype, (p0 || p1) ? (int)param_dtype : 0, vec};
    TwoPassArgs a{};  // aux (per-row outputs) stays null: these operators write none
    a.x = x; a.y = y; a.p0 = p0; a.p1 = p1;
    a.cols = cols;
    a.chunk = (int32_t)plan.slice_elems;
    a.nch = (int32_t)((cols + plan.slice_elems - 1) / plan.slice_elems);
    a.eps = eps;
    a.ws = static_cast<float*>(scratch);
    // The stats kernel writes every partial the apply kernel reads, so the
    // array needs no clearing between calls.
    const cudaError_t e = launch_two_pass(key, a, rows, plan.threads, (cudaStream_t)stream);
    return e == cudaSuccess ? CREDIT_OK : CREDIT_ERR_CUDA;
}
