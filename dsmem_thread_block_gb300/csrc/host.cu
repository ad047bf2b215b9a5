// host.cu -- operator calls on host buffers, pipelined over row chunks.
//
// A call whose inputs and outputs live in host memory is split into chunks of
// rows.  Three library-owned streams per device carry the host-to-device
// copies, the operator launches and the device-to-host copies; two device
// slots (inputs, output, per-row results) alternate between chunks, so chunk
// c's input copy, chunk c-1's kernel and chunk c-2's output copy run at the
// same time, and the two copy directions overlap each other.  Events order a
// slot's reuse: a chunk's input copy waits for the kernel that last read the
// slot, its kernel for the output copy that last read the slot's output.
// The call is stream-ordered like the device-buffer calls: the internal
// streams wait for the caller's stream at entry and the caller's stream waits
// for the last output copy at exit; nothing synchronises the host.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "credit.h"
#include "internal.h"
#include "planner.h"

namespace credit {
namespace {

constexpr int kSlots = 2;

struct HostPipe {
    bool ready = false;
    cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
    cudaEvent_t entry = nullptr;
    cudaEvent_t in_done[kSlots] = {}, comp_done[kSlots] = {}, out_done[kSlots] = {};
};

std::mutex g_host_mu;
HostPipe g_pipe[kMaxDevices];

// The device's streams and events, created once (caller holds g_host_mu).
HostPipe* host_pipe(int dev) {
    HostPipe& p = g_pipe[dev];
    if (p.ready) return &p;
    auto ev = [](cudaEvent_t* e) {
        return cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
    };
    bool ok = cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p.comp, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking) == cudaSuccess &&
              ev(&p.entry);
    for (int s = 0; ok && s < kSlots; ++s)
        ok = ev(&p.in_done[s]) && ev(&p.comp_done[s]) && ev(&p.out_done[s]);
    if (!ok) {
        cudaGetLastError();
        return nullptr;
    }
    p.ready = true;
    return &p;
}

int64_t round256(int64_t b) { return (b + 255) / 256 * 256; }

bool dtype_ok(credit_dtype_t d) { return d == CREDIT_F32 || d == CREDIT_BF16; }

// Byte sizes of one slot's regions for `rpc` rows.
struct SlotLayout {
    int64_t x, u, y, aux, slot, ws;
};

bool layout(const credit_host_call_t& c, const credit_plan_t* plan, int64_t rpc, SlotLayout* L) {
    if (!dtype_ok(c.dtype) || c.cols < 1 || rpc < 1) return false;
    const int64_t es = c.dtype == CREDIT_F32 ? 4 : 2;
    if (rpc > INT64_MAX / c.cols / es) return false;
    const int64_t mat = rpc * c.cols * es;
    L->x = round256(mat);
    L->u = c.op == CREDIT_PEARSON ? round256(mat) : 0;
    L->y = round256(c.op == CREDIT_QUANTIZE ? rpc * c.cols : mat);
    L->aux = (c.op == CREDIT_QUANTIZE || c.op == CREDIT_PEARSON) ? round256(rpc * 4) : 0;
    L->slot = L->x + L->u + L->y + L->aux;
    L->ws = 0;
    if (plan && plan->variant == CREDIT_TWO_PASS && plan->slice_elems > 0) {
        const int64_t nch = (c.cols + plan->slice_elems - 1) / plan->slice_elems;
        L->ws = round256(rpc * nch * (c.op == CREDIT_PEARSON ? 32 : 16));
    }
    return true;
}

// One operator launch on device pointers through the public entry points.
credit_status_t launch(const credit_host_call_t& c, const void* x, const void* u, void* y,
                       float* aux, int64_t rows, const credit_plan_t* plan, void* ws, size_t wsb,
                       cudaStream_t s) {
    switch (c.op) {
        case CREDIT_SOFTMAX: return credit_softmax(x, y, rows, c.cols, c.dtype, plan, ws, wsb, s);
        case CREDIT_LAYERNORM:
            return credit_layernorm(x, y, rows, c.cols, c.dtype, c.p0, c.p1, c.param_dtype, c.eps,
                                    plan, ws, wsb, s);
        case CREDIT_RMSNORM:
            return credit_rmsnorm(x, y, rows, c.cols, c.dtype, c.p0, c.param_dtype, c.eps, plan, ws,
                                  wsb, s);
        case CREDIT_QUANTIZE:
            return credit_quantize(x, static_cast<int8_t*>(y), aux, rows, c.cols, c.dtype, plan, ws,
                                   wsb, s);
        case CREDIT_WEIGHTED_STD:
            return credit_weighted_std(x, y, rows, c.cols, c.dtype, c.p0, c.param_dtype, c.eps,
                                       plan, ws, wsb, s);
        case CREDIT_PEARSON:
            return credit_pearson(x, u, y, aux, rows, c.cols, c.dtype, c.eps, plan, ws, wsb, s);
    }
    return CREDIT_ERR_UNSUPPORTED;
}

}  // namespace
}  // namespace credit

using namespace credit;

extern "C" credit_status_t credit_host_buffer_bytes(const credit_host_call_t* call,
                                                    const credit_plan_t* plan,
                                                    int64_t rows_per_chunk, size_t* bytes) {
    if (!call || !bytes) return CREDIT_ERR_INVALID_ARG;
    SlotLayout L;
    if (!layout(*call, plan, rows_per_chunk, &L)) return CREDIT_ERR_INVALID_ARG;
    *bytes = (size_t)(kSlots * L.slot + L.ws);
    return CREDIT_OK;
}

extern "C" credit_status_t credit_run_host(const credit_host_call_t* call,
                                           const credit_plan_t* plan, void* device_buffer,
                                           size_t device_buffer_bytes, int64_t rows_per_chunk,
                                           void* stream) {
    if (!call || !plan || !call->x || !call->y || call->rows < 1 || call->cols < 1 ||
        rows_per_chunk < 1)
        return CREDIT_ERR_INVALID_ARG;
    const credit_host_call_t& c = *call;
    const bool quant = c.op == CREDIT_QUANTIZE, pearson = c.op == CREDIT_PEARSON;
    if ((quant || pearson) && !c.row_out) return CREDIT_ERR_INVALID_ARG;
    if (pearson && !c.u) return CREDIT_ERR_INVALID_ARG;
    const int64_t rpc = rows_per_chunk < c.rows ? rows_per_chunk : c.rows;
    SlotLayout L;
    if (!layout(c, plan, rpc, &L)) return CREDIT_ERR_INVALID_ARG;
    if (!device_buffer || ((uintptr_t)device_buffer & 255u) ||
        device_buffer_bytes < (size_t)(kSlots * L.slot + L.ws))
        return CREDIT_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return CREDIT_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_host_mu);
    HostPipe* p = host_pipe(dev);
    if (!p) return CREDIT_ERR_CUDA;
    const cudaStream_t user = (cudaStream_t)stream;
    const int64_t es = c.dtype == CREDIT_F32 ? 4 : 2;
    const int64_t yes = quant ? 1 : es;
    unsigned char* base = static_cast<unsigned char*>(device_buffer);
    void* ws = L.ws ? base + kSlots * L.slot : nullptr;

    // the pipeline starts after the caller's earlier work
    if (cudaEventRecord(p->entry, user) != cudaSuccess ||
        cudaStreamWaitEvent(p->h2d, p->entry, 0) != cudaSuccess ||
        cudaStreamWaitEvent(p->comp, p->entry, 0) != cudaSuccess ||
        cudaStreamWaitEvent(p->d2h, p->entry, 0) != cudaSuccess) {
        cudaGetLastError();
        return CREDIT_ERR_CUDA;
    }
    const int64_t nchunks = (c.rows + rpc - 1) / rpc;
    credit_status_t st = CREDIT_OK;
    int last = 0;
    for (int64_t k = 0; k < nchunks && st == CREDIT_OK; ++k) {
        const int s = (int)(k % kSlots);
        last = s;
        const int64_t r0 = k * rpc;
        const int64_t nr = c.rows - r0 < rpc ? c.rows - r0 : rpc;
        unsigned char* slot = base + s * L.slot;
        unsigned char* dx = slot;
        unsigned char* du = slot + L.x;
        unsigned char* dy = slot + L.x + L.u;
        float* daux = L.aux ? reinterpret_cast<float*>(slot + L.x + L.u + L.y) : nullptr;
        const size_t in_bytes = (size_t)(nr * c.cols * es);
        const size_t out_bytes = (size_t)(nr * c.cols * yes);
        const unsigned char* hx = static_cast<const unsigned char*>(c.x) + r0 * c.cols * es;
        cudaError_t e = cudaSuccess;
        // inputs, once the kernel that last read this slot is done
        if (k >= kSlots) e = cudaStreamWaitEvent(p->h2d, p->comp_done[s], 0);
        if (e == cudaSuccess) e = cudaMemcpyAsync(dx, hx, in_bytes, cudaMemcpyHostToDevice, p->h2d);
        if (e == cudaSuccess && pearson)
            e = cudaMemcpyAsync(du, static_cast<const unsigned char*>(c.u) + r0 * c.cols * es,
                                in_bytes, cudaMemcpyHostToDevice, p->h2d);
        if (e == cudaSuccess) e = cudaEventRecord(p->in_done[s], p->h2d);
        // the kernel, once its inputs are in and the slot's last output is out
        if (e == cudaSuccess) e = cudaStreamWaitEvent(p->comp, p->in_done[s], 0);
        if (e == cudaSuccess && k >= kSlots) e = cudaStreamWaitEvent(p->comp, p->out_done[s], 0);
        if (e != cudaSuccess) { cudaGetLastError(); st = CREDIT_ERR_CUDA; break; }
        st = launch(c, dx, pearson ? du : nullptr, dy, daux, nr, plan, ws, (size_t)L.ws, p->comp);
        if (st != CREDIT_OK) break;
        e = cudaEventRecord(p->comp_done[s], p->comp);
        // the outputs
        if (e == cudaSuccess) e = cudaStreamWaitEvent(p->d2h, p->comp_done[s], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(static_cast<unsigned char*>(c.y) + r0 * c.cols * yes, dy, out_bytes,
                                cudaMemcpyDeviceToHost, p->d2h);
        if (e == cudaSuccess && daux)
            e = cudaMemcpyAsync(c.row_out + r0, daux, (size_t)(nr * 4), cudaMemcpyDeviceToHost,
                                p->d2h);
        if (e == cudaSuccess) e = cudaEventRecord(p->out_done[s], p->d2h);
        if (e != cudaSuccess) { cudaGetLastError(); st = CREDIT_ERR_CUDA; }
    }
    // the caller's stream resumes after the last output copy (the d2h stream
    // is in order, so that covers every chunk) -- also after a failure, so
    // that nothing the pipeline enqueued outlives the call's stream order
    if (cudaStreamWaitEvent(user, p->out_done[last], 0) != cudaSuccess ||
        cudaStreamWaitEvent(user, p->comp_done[last], 0) != cudaSuccess ||
        cudaStreamWaitEvent(user, p->in_done[last], 0) != cudaSuccess) {
        cudaGetLastError();
        if (st == CREDIT_OK) st = CREDIT_ERR_CUDA;
    }
    return st;
}
