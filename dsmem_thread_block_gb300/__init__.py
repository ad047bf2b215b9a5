"""GB300-native CREDIT reduce-reuse library.

Clustered DSMEM row softmax, LayerNorm, RMSNorm, int8 quantization, weighted
standardization and Pearson correlation behind a C ABI
(``libcredit.so``, declared in ``include/credit.h``), with this thin torch
binding on top.  The binding only marshals arguments (device pointers, sizes,
the current CUDA stream, a workspace from torch's allocator); every step of
the computation runs in the library's CUDA kernels, and a missing library
raises instead of falling back to anything else.

    import torch, dsmem_thread_block_gb300 as credit
    y = credit.layernorm(x, gamma, beta, eps=1e-5)       # plans automatically
    p = credit.plan("softmax", rows, cols, torch.float32, cluster_size=4)
    y = credit.softmax(x, plan=p)                         # forced cluster size
"""
from __future__ import annotations

from . import _credit as C
from ._credit import CreditError, Plan  # noqa: F401

__all__ = ["softmax", "layernorm", "rmsnorm", "quantize", "weighted_std", "pearson", "plan",
           "CreditError", "Plan", "device_error", "load_library"]

_OPS = {"softmax": C.SOFTMAX, "layernorm": C.LAYERNORM, "rmsnorm": C.RMSNORM,
        "quantize": C.QUANTIZE, "weighted_std": C.WEIGHTED_STD, "pearson": C.PEARSON}
_plan_cache: dict = {}


def load_library():
    """Load libcredit.so (raises if it has not been built)."""
    return C.load()


def _dtype(t):
    import torch
    if t == torch.float32:
        return C.F32
    if t == torch.bfloat16:
        return C.BF16
    raise TypeError(f"credit: unsupported dtype {t} (fp32 and bf16 only)")


def plan(op: str, rows: int, cols: int, dtype, device: int | None = None,
         variant: str | None = None, cluster_size: int = 1, rows_per_cluster: int = 0,
         exchange: str | None = None, staged_elems: int = 0) -> Plan:
    """Plan a call: automatically (variant None) or for a forced variant
    ("cluster" with `cluster_size` and optionally `rows_per_cluster` or
    `staged_elems` (an L2-tail plan staging that many elements of each
    slice), "persistent" or "pipelined" with `cluster_size`, "warp_rows" or
    "two_pass"); `exchange` ("async" or "barrier") picks how a clustered plan
    exchanges its partials."""
    import torch
    dev = torch.cuda.current_device() if device is None else int(device)
    code = _OPS[op]
    if variant is None:
        return C.credit_plan(code, rows, cols, _dtype(dtype), dev)
    v = {"cluster": C.CLUSTER, "persistent": C.CLUSTER_PERSISTENT,
         "pipelined": C.CLUSTER_PIPELINED, "warp_rows": C.WARP_ROWS,
         "two_pass": C.TWO_PASS}[variant]
    x = {None: C.EXCHANGE_DEFAULT, "async": C.EXCHANGE_ASYNC,
         "barrier": C.EXCHANGE_BARRIER}[exchange]
    return C.credit_plan_with(code, rows, cols, _dtype(dtype), dev, v, cluster_size,
                              rows_per_cluster=rows_per_cluster, exchange=x,
                              staged_elems=staged_elems)


def _prep(x, out):
    import torch
    if not x.is_cuda:
        raise ValueError("credit: x must be a CUDA tensor")
    if not x.is_contiguous():
        raise ValueError("credit: x must be contiguous")
    cols = x.shape[-1]
    rows = x.numel() // cols if cols else 0
    if out is None:
        out = torch.empty_like(x)
    elif out.shape != x.shape or out.dtype != x.dtype or not out.is_contiguous():
        raise ValueError("credit: out must be a contiguous tensor shaped like x")
    return rows, cols, out


def _plan_and_ws(op, rows, cols, x, p, workspace):
    import torch
    if p is None:
        key = (op, rows, cols, x.dtype, x.device.index)
        p = _plan_cache.get(key)
        if p is None:
            p = C.credit_plan(_OPS[op], rows, cols, _dtype(x.dtype), x.device.index)
            _plan_cache[key] = p
    need = int(p.workspace_bytes)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    wptr = workspace.data_ptr() if workspace is not None else 0
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return p, wptr, wbytes


def _stream(x):
    import torch
    return torch.cuda.current_stream(x.device).cuda_stream


def _ptr(t):
    return t.data_ptr() if t is not None else 0


def _pdtype(*ts):
    ts = [t for t in ts if t is not None]
    if not ts:
        return C.F32
    d = ts[0].dtype
    for t in ts:
        if t.dtype != d or not t.is_cuda or not t.is_contiguous():
            raise ValueError("credit: parameters must be contiguous CUDA tensors of one dtype")
    return _dtype(d)


def softmax(x, out=None, plan: Plan | None = None, workspace=None):
    """Row softmax over the last dimension."""
    rows, cols, out = _prep(x, out)
    p, w, wb = _plan_and_ws("softmax", rows, cols, x, plan, workspace)
    st = C.credit_softmax(x.data_ptr(), out.data_ptr(), rows, cols, _dtype(x.dtype), p, w, wb,
                          _stream(x))
    if st != C.OK:
        raise CreditError(st, "credit_softmax")
    return out


def layernorm(x, gamma=None, beta=None, eps: float = 1e-5, out=None, plan: Plan | None = None,
              workspace=None):
    """LayerNorm over the last dimension (biased variance, eps inside the sqrt)."""
    rows, cols, out = _prep(x, out)
    for t in (gamma, beta):
        if t is not None and t.numel() != cols:
            raise ValueError("credit: gamma/beta must have cols elements")
    p, w, wb = _plan_and_ws("layernorm", rows, cols, x, plan, workspace)
    st = C.credit_layernorm(x.data_ptr(), out.data_ptr(), rows, cols, _dtype(x.dtype),
                            _ptr(gamma), _ptr(beta), _pdtype(gamma, beta), float(eps), p, w, wb,
                            _stream(x))
    if st != C.OK:
        raise CreditError(st, "credit_layernorm")
    return out


def rmsnorm(x, weight=None, eps: float = 1e-6, out=None, plan: Plan | None = None,
            workspace=None):
    """RMSNorm over the last dimension."""
    rows, cols, out = _prep(x, out)
    if weight is not None and weight.numel() != cols:
        raise ValueError("credit: weight must have cols elements")
    p, w, wb = _plan_and_ws("rmsnorm", rows, cols, x, plan, workspace)
    st = C.credit_rmsnorm(x.data_ptr(), out.data_ptr(), rows, cols, _dtype(x.dtype),
                          _ptr(weight), _pdtype(weight), float(eps), p, w, wb, _stream(x))
    if st != C.OK:
        raise CreditError(st, "credit_rmsnorm")
    return out


def quantize(x, out=None, scales=None, plan: Plan | None = None, workspace=None):
    """Row-wise symmetric int8 quantization over the last dimension; returns
    (codes int8 shaped like x, fp32 scales, one per row)."""
    import torch
    if not x.is_cuda or not x.is_contiguous():
        raise ValueError("credit: x must be a contiguous CUDA tensor")
    cols = x.shape[-1]
    rows = x.numel() // cols if cols else 0
    if out is None:
        out = torch.empty(x.shape, dtype=torch.int8, device=x.device)
    if scales is None:
        scales = torch.empty(rows, dtype=torch.float32, device=x.device)
    p, w, wb = _plan_and_ws("quantize", rows, cols, x, plan, workspace)
    st = C.credit_quantize(x.data_ptr(), out.data_ptr(), scales.data_ptr(), rows, cols,
                           _dtype(x.dtype), p, w, wb, _stream(x))
    if st != C.OK:
        raise CreditError(st, "credit_quantize")
    return out, scales


def weighted_std(x, weights, eps: float = 1e-5, out=None, plan: Plan | None = None,
                 workspace=None):
    """Weighted standardization over the last dimension with per-column
    weights: (x - mean_w) / sqrt(var_w + eps)."""
    rows, cols, out = _prep(x, out)
    if weights is None or weights.numel() != cols:
        raise ValueError("credit: weights must have cols elements")
    p, w, wb = _plan_and_ws("weighted_std", rows, cols, x, plan, workspace)
    st = C.credit_weighted_std(x.data_ptr(), out.data_ptr(), rows, cols, _dtype(x.dtype),
                               weights.data_ptr(), _pdtype(weights), float(eps), p, w, wb,
                               _stream(x))
    if st != C.OK:
        raise CreditError(st, "credit_weighted_std")
    return out


def pearson(x, u, eps: float = 0.0, out=None, r=None, plan: Plan | None = None, workspace=None):
    """Row-wise Pearson correlation of x and u over the last dimension;
    returns (standardized co-deviations shaped like x, fp32 r per row)."""
    import torch
    rows, cols, out = _prep(x, out)
    if u is None or u.shape != x.shape or u.dtype != x.dtype or not u.is_cuda or \
            not u.is_contiguous():
        raise ValueError("credit: u must be a contiguous CUDA tensor shaped like x")
    if r is None:
        r = torch.empty(rows, dtype=torch.float32, device=x.device)
    p, w, wb = _plan_and_ws("pearson", rows, cols, x, plan, workspace)
    st = C.credit_pearson(x.data_ptr(), u.data_ptr(), out.data_ptr(), r.data_ptr(), rows, cols,
                          _dtype(x.dtype), float(eps), p, w, wb, _stream(x))
    if st != C.OK:
        raise CreditError(st, "credit_pearson")
    return out, r


def device_error(device: int = 0) -> int:
    """Read and clear the device error word (CREDIT_ERR_DEVICE_TIMEOUT if a
    bounded device wait gave up)."""
    return C.credit_get_device_error(device)
