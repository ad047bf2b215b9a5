"""Plain CPU oracle for row softmax, LayerNorm, RMSNorm, int8 quantization,
weighted standardization and Pearson correlation (fp64; the quantization
codes in IEEE single).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product library never loads it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, fp64, the textbook definitions
of the operators, cited there).  This module compiles it with gcc, loads it
with ctypes and wraps it for numpy arrays.  bf16 buffers travel as ``uint16``
arrays holding the raw bit patterns; the C side widens them exactly.

Parity pins: every function here is pinned by ``tests/test_oracle.py``
(closed forms, invariants, a library cross-check and hand-derived fixtures in
``tests/golden/``).
"""
from __future__ import annotations

import concurrent.futures as _cf
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")

F32, BF16, F64 = 0, 1, 2
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc -O2, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".{os.getpid()}.tmp"
    subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-Wall",
                    "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp,
                    "-lm"], check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, i64, i32, dbl = (ctypes.c_void_p, ctypes.c_int64,
                                 ctypes.c_int, ctypes.c_double)
            lib.oracle_widen.argtypes = [vp, i32, i64, vp]
            lib.oracle_softmax.argtypes = [vp, i32, i64, i64, vp]
            lib.oracle_layernorm.argtypes = [vp, i32, i64, i64, vp, vp, i32,
                                             dbl, vp, vp]
            lib.oracle_rmsnorm.argtypes = [vp, i32, i64, i64, vp, i32, dbl,
                                           vp]
            lib.oracle_quantize.argtypes = [vp, i32, i64, i64, vp, vp]
            lib.oracle_weighted_std.argtypes = [vp, i32, i64, i64, vp, i32, dbl, vp]
            lib.oracle_pearson.argtypes = [vp, vp, i32, i64, i64, dbl, vp, vp]
            for f in (lib.oracle_widen, lib.oracle_softmax, lib.oracle_layernorm,
                      lib.oracle_rmsnorm, lib.oracle_quantize, lib.oracle_weighted_std,
                      lib.oracle_pearson):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:  # raw bf16 bit patterns
        return BF16
    if a.dtype == np.float64:
        return F64
    raise TypeError(f"oracle: unsupported input dtype {a.dtype}")


def _ptr(a):
    return None if a is None else a.ctypes.data


def _prep(x: np.ndarray):
    x = np.ascontiguousarray(x)
    if x.ndim == 1:
        x = x.reshape(1, -1)
    if x.ndim != 2:
        raise ValueError("oracle: x must be 1-D or 2-D")
    return x


def _vec(v, cols):
    if v is None:
        return None, F32
    v = np.ascontiguousarray(v).reshape(-1)
    if v.shape[0] != cols:
        raise ValueError("oracle: parameter vector length != cols")
    return v, _dtype_code(v)


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"oracle: {name} rejected its arguments (rc={rc})")


def widen(x: np.ndarray) -> np.ndarray:
    """Exact fp64 value of every element of an fp32 / bf16(uint16) / fp64 array."""
    x = np.ascontiguousarray(x)
    out = np.empty(x.shape, dtype=np.float64)
    _check(_load().oracle_widen(_ptr(x), _dtype_code(x), x.size, _ptr(out)),
           "widen")
    return out


def softmax(x: np.ndarray) -> np.ndarray:
    x = _prep(x)
    y = np.empty(x.shape, dtype=np.float64)
    _check(_load().oracle_softmax(_ptr(x), _dtype_code(x), x.shape[0],
                                  x.shape[1], _ptr(y)), "softmax")
    return y


def layernorm(x: np.ndarray, gamma=None, beta=None, eps: float = 1e-5,
              want_z: bool = False):
    x = _prep(x)
    g, gd = _vec(gamma, x.shape[1])
    b, bd = _vec(beta, x.shape[1])
    if g is not None and b is not None and gd != bd:
        raise TypeError("oracle: gamma and beta must share a dtype")
    pd = gd if g is not None else bd
    y = np.empty(x.shape, dtype=np.float64)
    z = np.empty(x.shape, dtype=np.float64) if want_z else None
    _check(_load().oracle_layernorm(_ptr(x), _dtype_code(x), x.shape[0],
                                    x.shape[1], _ptr(g), _ptr(b), pd,
                                    float(eps), _ptr(y), _ptr(z)),
           "layernorm")
    return (y, z) if want_z else y


def rmsnorm(x: np.ndarray, weight=None, eps: float = 1e-6) -> np.ndarray:
    x = _prep(x)
    w, wd = _vec(weight, x.shape[1])
    y = np.empty(x.shape, dtype=np.float64)
    _check(_load().oracle_rmsnorm(_ptr(x), _dtype_code(x), x.shape[0],
                                  x.shape[1], _ptr(w), wd, float(eps),
                                  _ptr(y)), "rmsnorm")
    return y


def quantize(x: np.ndarray):
    """Row-wise symmetric int8 codes and fp32 scales (see oracle.c)."""
    x = _prep(x)
    q = np.empty(x.shape, dtype=np.int8)
    s = np.empty(x.shape[0], dtype=np.float32)
    _check(_load().oracle_quantize(_ptr(x), _dtype_code(x), x.shape[0], x.shape[1], _ptr(q),
                                   _ptr(s)), "quantize")
    return q, s


def weighted_std(x: np.ndarray, w: np.ndarray, eps: float = 1e-5) -> np.ndarray:
    """Row-wise weighted standardization with per-column weights (see oracle.c)."""
    x = _prep(x)
    wv, wd = _vec(w, x.shape[1])
    y = np.empty(x.shape, dtype=np.float64)
    _check(_load().oracle_weighted_std(_ptr(x), _dtype_code(x), x.shape[0], x.shape[1],
                                       _ptr(wv), wd, float(eps), _ptr(y)), "weighted_std")
    return y


def pearson(x: np.ndarray, u: np.ndarray, eps: float = 0.0):
    """Row-wise standardized co-deviations and correlations (see oracle.c):
    returns (y fp64 shaped like x, r fp64 one per row)."""
    x = _prep(x)
    u = _prep(u)
    if u.shape != x.shape or _dtype_code(u) != _dtype_code(x):
        raise ValueError("oracle: x and u must share shape and dtype")
    y = np.empty(x.shape, dtype=np.float64)
    r = np.empty(x.shape[0], dtype=np.float64)
    _check(_load().oracle_pearson(_ptr(x), _ptr(u), _dtype_code(x), x.shape[0], x.shape[1],
                                  float(eps), _ptr(y), _ptr(r)), "pearson")
    return y, r


def run_rows(fn, x: np.ndarray, *args, threads: int = 1, **kw) -> np.ndarray:
    """Apply a row-wise oracle function with the rows split over `threads`
    host threads.  The C calls release the GIL, so the threads run in
    parallel; each row is still computed by the same serial code."""
    x = _prep(x)
    if threads <= 1 or x.shape[0] <= 1:
        return fn(x, *args, **kw)
    bounds = np.linspace(0, x.shape[0], min(threads, x.shape[0]) + 1,
                         dtype=np.int64)
    out = np.empty(x.shape, dtype=np.float64)

    def part(i):
        lo, hi = int(bounds[i]), int(bounds[i + 1])
        out[lo:hi] = fn(x[lo:hi], *args, **kw)

    with _cf.ThreadPoolExecutor(max_workers=len(bounds) - 1) as ex:
        list(ex.map(part, range(len(bounds) - 1)))
    return out
