"""Planted slips in the oracle must fail its pins.

Each case copies the oracle package to a temporary directory, plants one
plausible mistake in oracle.c (a dropped max shift, an unbiased variance, eps
outside the square root, a row-indexed parameter, a swapped affine order, a
wrong bf16 widening, rounding ties away from zero, truncated codes, a wrong scale, an
unweighted sum, a transposed operand, a dropped eps or normaliser), rebuilds
it with gcc and runs the pin tests against it.  Every planted slip must make
at least one pin fail; the unmodified copy must pass.  Mistakes are planted in
the CPU oracle only.  (The quantization clamp at +-127 is not among them:
with scale = amax / 127 no finite quotient reaches +-127.5, so a changed
clamp changes no code.)
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, text in oracle.c, replacement)
SLIPS = [
    ("softmax without the max shift", "s += exp(or_load(x, dtype, base + j) - m);",
     "s += exp(or_load(x, dtype, base + j));"),
    ("softmax output not normalised", "y[base + j] = exp(or_load(x, dtype, base + j) - m) / s;",
     "y[base + j] = exp(or_load(x, dtype, base + j) - m) / (s + 1.0);"),
    ("unbiased LayerNorm variance", "var = ssd / (double)cols;", "var = ssd / (double)(cols - 1);"),
    ("eps outside the square root", "inv = 1.0 / sqrt(var + eps);\n        for (j = 0; j < cols; ++j) {\n            double zj",
     "inv = 1.0 / (sqrt(var) + eps);\n        for (j = 0; j < cols; ++j) {\n            double zj"),
    ("beta indexed by row", "double b = beta ? or_load(beta, pdtype, j) : 0.0;",
     "double b = beta ? or_load(beta, pdtype, r) : 0.0;"),
    ("affine steps swapped", "y[base + j] = zj * g + b;", "y[base + j] = (zj + b) * g;"),
    ("bf16 widened by 15 bits", "u = ((uint32_t)h) << 16;", "u = ((uint32_t)h) << 15;"),
    ("RMSNorm without eps", "inv = 1.0 / sqrt(ss / (double)cols + eps);",
     "inv = 1.0 / sqrt(ss / (double)cols);"),
    ("quantization ties away from zero", "c = rintf(v / s);", "c = roundf(v / s);"),
    ("quantization scale over 128", "s = (float)amax / 127.0f;", "s = (float)amax / 128.0f;"),
    ("quantization codes truncated", "c = rintf(v / s);", "c = truncf(v / s);"),
    ("unweighted mean", "sw += wj * or_load(x, dtype, base + j);",
     "sw += or_load(x, dtype, base + j);"),
    ("unweighted variance", "ssd += or_load(w, wdtype, j) * d * d;", "ssd += d * d;"),
    ("weighted variance over W - 1", "var = ssd / W;", "var = ssd / (W - 1.0);"),
    ("Pearson mean of u from x", "mu = su / (double)cols;", "mu = sx / (double)cols;"),
    ("Pearson covariance as a variance", "sxu += dx * du;", "sxu += dx * dx;"),
    ("Pearson eps dropped on one side",
     "den = sqrt((sxx / (double)cols + eps) * (suu / (double)cols + eps));",
     "den = sqrt((sxx / (double)cols) * (suu / (double)cols + eps));"),
    ("Pearson output with a transposed operand", "y[base + j] = dx * du / den;",
     "y[base + j] = du * du / den;"),
    ("Pearson r not divided by N", "r[i] = (sxu / (double)cols) / den;", "r[i] = sxu / den;"),
]


def _run_pins(tmp, src_text):
    pkg = os.path.join(tmp, "oracle")
    shutil.copytree(os.path.join(ROOT, "oracle"), pkg,
                    ignore=shutil.ignore_patterns("_build", "__pycache__"))
    with open(os.path.join(pkg, "oracle.c"), "w") as f:
        f.write(src_text)
    env = dict(os.environ, PYTHONPATH=tmp + os.pathsep + ROOT)
    # the pins import `oracle` from PYTHONPATH's first entry: the planted copy
    p = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "-m", "not gpu", os.path.join(ROOT, "tests", "test_oracle.py")],
                       env=env, cwd=tmp, capture_output=True, text=True, timeout=600)
    return p.returncode, p.stdout[-400:]


@pytest.fixture(scope="module")
def source():
    with open(os.path.join(ROOT, "oracle", "oracle.c")) as f:
        return f.read()


def test_unmodified_copy_passes(source, tmp_path):
    rc, out = _run_pins(str(tmp_path), source)
    assert rc == 0, out


@pytest.mark.parametrize("name,old,new", SLIPS, ids=[s[0] for s in SLIPS])
def test_planted_slip_fails_a_pin(source, tmp_path, name, old, new):
    assert source.count(old) == 1, f"slip text not found once: {name}"
    rc, out = _run_pins(str(tmp_path), source.replace(old, new))
    assert rc != 0, f"no pin caught: {name}\n{out}"
