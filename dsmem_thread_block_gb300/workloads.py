"""Seeded synthetic inputs for the wide-row reduce-then-reuse operators.

This module only draws numbers: it holds none of the operators' arithmetic and
imports neither the CUDA binding nor the oracle, so both sides can consume the
very same bytes.  All draws use numpy's PCG64 generator
(``numpy.random.default_rng(seed)``), which is deterministic across machines.
In ``N(mu, sigma)`` the second parameter is the standard deviation.  bf16
tensors are rounded from the fp32 draws to nearest-even (torch's cast) and
returned as ``uint16`` arrays holding the raw bit patterns.

The shapes follow the CREDIT page's wide-reduction workloads (section
"A. Experimental Setup and Baselines": thousands of rows, widths of 4K and
wider, FP32) widened to rows that no single SM can stage.
"""
from __future__ import annotations

import dataclasses

import numpy as np

SOFTMAX, LAYERNORM, RMSNORM = "softmax", "layernorm", "rmsnorm"
QUANTIZE, WEIGHTED_STD, PEARSON = "quantize", "weighted_std", "pearson"


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest-even) and return the raw bits."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact fp32 value of raw bf16 bit patterns (zero-extend the mantissa)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32)
            << 16).view(np.float32)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic problem: op, element type, shape and input recipe."""
    name: str
    op: str
    dtype: str                  # "f32" or "bf16" (input and output)
    rows: int
    cols: int
    seed: int
    x_mean: float = 0.0
    x_std: float = 1.0
    spike_frac: float = 0.0     # softmax stress: fraction of entries set to spike_value
    spike_value: float = 30.0
    eps: float = 0.0
    param_dtype: str | None = None   # dtype of gamma/beta or weight, None = no params
    p_mean: float = 1.0         # gamma / weight ~ N(p_mean, p_std)
    p_std: float = 0.1
    b_mean: float = 0.0         # beta ~ N(b_mean, b_std)
    b_std: float = 0.1
    p_uniform: bool = False     # parameters ~ U(0, 1) instead (weights of weighted_std)
    u_corr: float = 0.6         # Pearson: u = u_corr * x + sqrt(1 - u_corr^2) * N(0, 1)

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def with_rows(self, rows: int) -> "Workload":
        return dataclasses.replace(self, rows=rows, name=f"{self.name}[rows={rows}]")

    def ideal_bytes(self) -> int:
        """One read plus one write of the matrix, parameter vectors once
        (quantization writes one byte per element plus a scale per row)."""
        if self.op == QUANTIZE:
            return self.rows * self.cols * (self.elem_bytes + 1) + 4 * self.rows
        if self.op == PEARSON:  # x and u read, y written, one r per row
            return 3 * self.rows * self.cols * self.elem_bytes + 4 * self.rows
        b = 2 * self.rows * self.cols * self.elem_bytes
        if self.param_dtype is not None:
            pb = 4 if self.param_dtype == "f32" else 2
            nvec = 2 if self.op == LAYERNORM else 1
            b += nvec * self.cols * pb
        return b

    def generate(self) -> dict:
        """Draw x (then u, or gamma/beta or weight) in a fixed order from `seed`."""
        rng = np.random.default_rng(self.seed)
        n = self.rows * self.cols
        x = rng.standard_normal(n, dtype=np.float32)
        if self.x_std != 1.0:
            x *= np.float32(self.x_std)
        if self.x_mean != 0.0:
            x += np.float32(self.x_mean)
        if self.spike_frac > 0.0:
            mask = rng.random(n, dtype=np.float32) < self.spike_frac
            x[mask] = np.float32(self.spike_value)
        out = {}
        if self.op == PEARSON:
            e = rng.standard_normal(n, dtype=np.float32)
            u = np.float32(self.u_corr) * x + np.float32(np.sqrt(1.0 - self.u_corr ** 2)) * e
            u = u.reshape(self.rows, self.cols)
            out["u"] = u if self.dtype == "f32" else to_bf16_bits(u)
        if self.param_dtype is not None:
            if self.p_uniform:
                g = rng.random(self.cols, dtype=np.float32)
            else:
                g = rng.standard_normal(self.cols, dtype=np.float32) * \
                    np.float32(self.p_std) + np.float32(self.p_mean)
            if self.op == LAYERNORM:
                b = rng.standard_normal(self.cols, dtype=np.float32) * \
                    np.float32(self.b_std) + np.float32(self.b_mean)
            conv = (lambda a: a) if self.param_dtype == "f32" else to_bf16_bits
            if self.op == LAYERNORM:
                out["gamma"], out["beta"] = conv(g), conv(b)
            else:
                out["weight"] = conv(g)
        x = x.reshape(self.rows, self.cols)
        out["x"] = x if self.dtype == "f32" else to_bf16_bits(x)
        return out


# The five workloads.  Names describe what they are.
SOFTMAX_F32_64x4096 = Workload(
    "softmax_f32_64x4096", SOFTMAX, "f32", 64, 4096, seed=0)
LAYERNORM_BF16_1024x262144 = Workload(
    "layernorm_bf16_1024x262144", LAYERNORM, "bf16", 1024, 262144, seed=1,
    x_mean=0.5, x_std=2.0, eps=1e-5, param_dtype="f32")
SOFTMAX_F32_512x131072_SPIKES = Workload(
    "softmax_f32_512x131072_spikes", SOFTMAX, "f32", 512, 131072, seed=2,
    x_std=4.0, spike_frac=0.01, spike_value=30.0)
RMSNORM_BF16_2048x786432 = Workload(
    "rmsnorm_bf16_2048x786432", RMSNORM, "bf16", 2048, 786432, seed=3,
    eps=1e-6, param_dtype="bf16")

SWEEP_ELEMENTS = 1 << 28
SWEEP_COLS = [1 << k for k in range(10, 21)]


def sweep_point(cols: int) -> Workload:
    """bf16 softmax with 2^28 elements in total, `cols` wide."""
    return Workload(f"softmax_bf16_sweep_{cols}", SOFTMAX, "bf16",
                    SWEEP_ELEMENTS // cols, cols, seed=4)


# the pages' FP32 widths (4K-64K, 4,096 rows) at the widest point
QUANTIZE_F32_4096x65536 = Workload(
    "quantize_f32_4096x65536", QUANTIZE, "f32", 4096, 65536, seed=5)
WEIGHTED_STD_F32_4096x65536 = Workload(
    "weighted_std_f32_4096x65536", WEIGHTED_STD, "f32", 4096, 65536, seed=6, x_mean=0.5,
    x_std=2.0, eps=1e-5, param_dtype="f32", p_uniform=True)

PEARSON_F32_4096x65536 = Workload(
    "pearson_f32_4096x65536", PEARSON, "f32", 4096, 65536, seed=7, x_mean=0.5, x_std=2.0,
    eps=1e-5)

ALL = [SOFTMAX_F32_64x4096, LAYERNORM_BF16_1024x262144,
       SOFTMAX_F32_512x131072_SPIKES, RMSNORM_BF16_2048x786432,
       QUANTIZE_F32_4096x65536, WEIGHTED_STD_F32_4096x65536, PEARSON_F32_4096x65536]
