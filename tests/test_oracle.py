"""Pins for the fp64 CPU oracle (no GPU needed).

Each test fixes the oracle to something other than itself: hand-derived
closed forms (tests/golden/closed_forms.json), invariants that the operators'
definitions imply, special cases that reduce to a library routine, and an
independent library cross-check (torch fp64 on CPU).  The set is chosen so
that a plausible slip -- a dropped max shift, a dropped eps, an unbiased
variance, eps outside the square root, gamma/beta indexed by row, a swapped
affine order, a wrong bf16 widening -- fails at least one test.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import scipy.special

import oracle
from dsmem_thread_block_gb300 import workloads as wl


def _frac(s):
    return float(Fraction(s))


# ---------------------------------------------------------------- dtype widening
def test_bf16_widening_matches_fixture(golden):
    g = golden["bf16_bits"]
    bits = np.array([int(b, 16) for b in g["bits"]], dtype=np.uint16)
    got = oracle.widen(bits)
    want = [float(v) if v != "1/2" else 0.5 for v in g["values"]]
    assert got.tolist() == want
    assert math.copysign(1.0, got[6]) == -1.0  # -0 keeps its sign


def test_fp32_widening_is_exact():
    x = np.array([1.0, -2.5, 3.1415927, 1e-30, 6.0e37], dtype=np.float32)
    assert oracle.widen(x).tolist() == [float(v) for v in x]


# ---------------------------------------------------------------------- softmax
def test_softmax_ln_k_closed_form(golden):
    g = golden["softmax_ln_k"]
    x = np.log(np.array(g["k"], dtype=np.float64))
    y = oracle.softmax(x)[0]
    want = np.array([_frac(s) for s in g["expected"]])
    np.testing.assert_allclose(y, want, rtol=1e-14, atol=0)


def test_softmax_two_point_is_logistic(golden):
    g = golden["softmax_two_point"]
    bits = np.array([int(b, 16) for b in g["bf16_bits"]], dtype=np.uint16)
    y = oracle.softmax(bits)[0]
    want = scipy.special.expit(np.array(g["logistic_args"]))
    np.testing.assert_allclose(y, want, rtol=1e-15, atol=0)


def test_softmax_rows_sum_to_one_and_are_positive():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((7, 333)) * 5).astype(np.float32)
    y = oracle.softmax(x)
    assert (y > 0).all()
    np.testing.assert_allclose(y.sum(axis=1), 1.0, rtol=0, atol=1e-12)


def test_softmax_shift_invariance_exact_inputs():
    # k/256 + 1024 is exact in fp32 (18 significant bits), so the shifted
    # input is exactly x + 1024 and the outputs must agree.
    rng = np.random.default_rng(12)
    k = rng.integers(-2000, 2000, size=(3, 100))
    x = (k / 256.0).astype(np.float32)
    for c in (1024.0, -1024.0):
        xs = (k / 256.0 + c).astype(np.float32)
        assert np.array_equal(xs.astype(np.float64), x.astype(np.float64) + c)
        np.testing.assert_allclose(oracle.softmax(xs), oracle.softmax(x),
                                   rtol=1e-12, atol=0)


def test_softmax_large_logits_do_not_overflow():
    # exp(800) overflows fp64: only a max-shifted softmax stays finite.
    x = np.array([[800.0, 799.0, 798.0]])
    y = oracle.softmax(x)[0]
    want = oracle.softmax(np.array([[2.0, 1.0, 0.0]]))[0]
    assert np.isfinite(y).all()
    np.testing.assert_allclose(y, want, rtol=1e-14)


def test_softmax_constant_row_is_uniform():
    for n in (1, 8, 1024):
        y = oracle.softmax(np.full((2, n), -3.25, dtype=np.float32))
        assert (y == 1.0 / n).all()


def test_softmax_permutation_equivariance():
    rng = np.random.default_rng(13)
    x = rng.standard_normal((4, 57)).astype(np.float32)
    perm = rng.permutation(57)
    np.testing.assert_allclose(oracle.softmax(x[:, perm]),
                               oracle.softmax(x)[:, perm], rtol=1e-14)


def test_softmax_rows_are_independent():
    # each row of a non-square batch equals the closed form of that row alone
    k = np.arange(1, 9, dtype=np.float64)
    x = np.stack([np.log(k), np.log(k[::-1]), np.zeros(8)])
    y = oracle.softmax(x)
    np.testing.assert_allclose(y[0], k / 36, rtol=1e-14)
    np.testing.assert_allclose(y[1], k[::-1] / 36, rtol=1e-14)
    np.testing.assert_allclose(y[2], 1 / 8, rtol=1e-15)


# -------------------------------------------------------------------- layernorm
def test_layernorm_1_to_8_closed_form(golden):
    g = golden["layernorm_1_to_8"]
    x = np.array(g["x"], dtype=np.float32)
    mu, var = _frac(g["mean"]), _frac(g["var"])
    eps = 0.25  # large enough that eps placement matters
    gamma = np.arange(1, 9, dtype=np.float32)       # gamma_j = j
    beta = -np.arange(1, 9, dtype=np.float32) / 4   # beta_j = -j/4
    y = oracle.layernorm(x, gamma, beta, eps=eps)[0]
    z = (np.array(g["x"]) - mu) / math.sqrt(var + eps)
    want = z * np.arange(1, 9) - np.arange(1, 9) / 4
    np.testing.assert_allclose(y, want, rtol=1e-14, atol=1e-15)


def test_layernorm_moments_without_affine():
    rng = np.random.default_rng(21)
    x = (rng.standard_normal((5, 1000)) * 3 + 7).astype(np.float32)
    xd = x.astype(np.float64)
    var = xd.var(axis=1)
    for eps in (0.0, 1e-5, 0.5):
        y = oracle.layernorm(x, eps=eps)
        np.testing.assert_allclose(y.mean(axis=1), 0.0, atol=1e-12)
        np.testing.assert_allclose(y.var(axis=1), var / (var + eps),
                                   rtol=1e-12)


def test_layernorm_scale_shift_invariance_eps0():
    rng = np.random.default_rng(22)
    k = rng.integers(-500, 500, size=(3, 64)).astype(np.float64)
    x = k / 16.0
    y0 = oracle.layernorm(x, eps=0.0)
    y1 = oracle.layernorm(x * 4.0 + 256.0, eps=0.0)
    np.testing.assert_allclose(y1, y0, rtol=1e-12, atol=1e-13)


def test_layernorm_constant_row_gives_beta():
    beta = np.linspace(-1, 1, 16).astype(np.float32)
    gamma = np.full(16, 3.0, dtype=np.float32)
    y = oracle.layernorm(np.full((2, 16), 0.75, dtype=np.float32),
                         gamma, beta, eps=1e-5)
    assert (y == beta.astype(np.float64)).all()


def test_layernorm_params_index_columns_not_rows():
    rng = np.random.default_rng(23)
    x = rng.standard_normal((3, 5)).astype(np.float32)
    gamma = np.array([1, 2, 3, 4, 5], dtype=np.float32)
    beta = np.array([0, 10, 20, 30, 40], dtype=np.float32)
    y, z = oracle.layernorm(x, gamma, beta, eps=1e-5, want_z=True)
    np.testing.assert_allclose(y, z * gamma + beta, rtol=1e-15, atol=1e-14)
    z_alone = oracle.layernorm(x, eps=1e-5)
    np.testing.assert_allclose(z, z_alone, rtol=0, atol=0)


# ---------------------------------------------------------------------- rmsnorm
def test_rmsnorm_1_to_8_closed_form(golden):
    g = golden["rmsnorm_1_to_8"]
    x = np.array(g["x"], dtype=np.float32)
    ms = _frac(g["mean_square"])
    eps = 0.5
    w = (2.0 ** -np.arange(8)).astype(np.float32)
    y = oracle.rmsnorm(x, w, eps=eps)[0]
    want = np.array(g["x"]) / math.sqrt(ms + eps) * (2.0 ** -np.arange(8))
    np.testing.assert_allclose(y, want, rtol=1e-15)


def test_rmsnorm_output_rms():
    rng = np.random.default_rng(31)
    x = (rng.standard_normal((4, 777)) * 2).astype(np.float32)
    ms = (x.astype(np.float64) ** 2).mean(axis=1)
    for eps in (0.0, 1e-6, 2.0):
        y = oracle.rmsnorm(x, eps=eps)
        np.testing.assert_allclose(np.sqrt((y ** 2).mean(axis=1)),
                                   np.sqrt(ms / (ms + eps)), rtol=1e-12)


# ------------------------------------------------- independent library routine
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_oracle_matches_torch_fp64(dtype):
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(41)
    x32 = (rng.standard_normal((6, 203)) * 2 + 0.5).astype(np.float32)
    x = x32 if dtype == "f32" else wl.to_bf16_bits(x32)
    xd = torch.from_numpy(oracle.widen(x))
    g = (rng.standard_normal(203) * 0.1 + 1).astype(np.float32)
    b = (rng.standard_normal(203) * 0.1).astype(np.float32)
    gt, bt = torch.from_numpy(g).double(), torch.from_numpy(b).double()
    np.testing.assert_allclose(oracle.softmax(x), F.softmax(xd, dim=1).numpy(),
                               rtol=1e-12, atol=0)
    np.testing.assert_allclose(
        oracle.layernorm(x, g, b, eps=1e-5),
        F.layer_norm(xd, (203,), gt, bt, eps=1e-5).numpy(), rtol=1e-11,
        atol=1e-13)
    np.testing.assert_allclose(
        oracle.rmsnorm(x, g, eps=1e-6),
        F.rms_norm(xd, (203,), gt, eps=1e-6).numpy(), rtol=1e-12, atol=1e-14)


def test_bf16_params_widen_exactly():
    rng = np.random.default_rng(42)
    x = rng.standard_normal((2, 64)).astype(np.float32)
    w32 = (rng.standard_normal(64) * 0.1 + 1).astype(np.float32)
    wb = wl.to_bf16_bits(w32)
    np.testing.assert_array_equal(oracle.rmsnorm(x, wb, eps=1e-6),
                                  oracle.rmsnorm(x, wl.bf16_bits_to_f32(wb),
                                                 eps=1e-6))


def test_threaded_rows_equal_serial():
    rng = np.random.default_rng(43)
    x = rng.standard_normal((37, 129)).astype(np.float32)
    np.testing.assert_array_equal(oracle.run_rows(oracle.softmax, x, threads=4),
                                  oracle.softmax(x))


def test_oracle_rejects_bad_arguments():
    with pytest.raises(TypeError):
        oracle.softmax(np.zeros((2, 2), dtype=np.int32))
    with pytest.raises(ValueError):
        oracle.rmsnorm(np.zeros((2, 4), np.float32), np.ones(3, np.float32))
    with pytest.raises(ValueError):
        oracle.layernorm(np.zeros((1, 4), np.float32), eps=-1.0)


# ------------------------------------------------------------------ generators
def test_workload_generators_are_seeded_and_shaped():
    w = wl.LAYERNORM_BF16_1024x262144.with_rows(2)
    a, b = w.generate(), w.generate()
    assert a["x"].dtype == np.uint16 and a["x"].shape == (2, 262144)
    assert np.array_equal(a["x"], b["x"]) and np.array_equal(a["gamma"], b["gamma"])
    xf = wl.bf16_bits_to_f32(a["x"])
    assert abs(float(xf.mean()) - 0.5) < 0.02 and abs(float(xf.std()) - 2.0) < 0.02
    s = wl.SOFTMAX_F32_512x131072_SPIKES.with_rows(2).generate()["x"]
    frac = float((s == 30.0).mean())
    assert 0.008 < frac < 0.012
    assert wl.sweep_point(1024).rows * 1024 == 1 << 28
    pr = wl.PEARSON_F32_4096x65536.with_rows(2).generate()
    assert pr["u"].shape == pr["x"].shape == (2, 65536)
    _, r = oracle.pearson(pr["x"], pr["u"])
    # u = 0.6 x + 0.8 e with std(x) = 2: r = 1.2 / sqrt(1.44 + 0.64) ~ 0.832
    assert np.all(np.abs(r - 1.2 / math.sqrt(2.08)) < 0.01)


# ----------------------------------------------------------------- quantization
def test_quantize_power_of_two_closed_form(golden):
    g = golden["quantize_power_of_two"]
    q, s = oracle.quantize(np.array(g["x"], dtype=np.float32))
    assert q[0].tolist() == g["q"] and s[0] == _frac(g["scale"])


def test_quantize_invariants():
    rng = np.random.default_rng(51)
    x = (rng.standard_normal((6, 999)) * 3).astype(np.float32)
    q, s = oracle.quantize(x)
    assert (np.abs(q) <= 127).all()
    # the absmax element maps to +-127, and the codes reconstruct x to half a step
    i = np.abs(x).argmax(axis=1)
    assert (np.abs(q[np.arange(6), i]) == 127).all()
    np.testing.assert_array_less(np.abs(q * s[:, None].astype(np.float64) - x) - 0.5 * s[:, None] * 1.0001, 0)
    # odd symmetry and exact scaling by powers of two
    qn, sn = oracle.quantize(-x)
    assert (qn == -q).all() and (sn == s).all()
    q4, s4 = oracle.quantize(x * np.float32(4))
    assert (q4 == q).all() and (s4 == 4 * s).all()


def test_quantize_zero_row_and_bf16_input():
    q, s = oracle.quantize(np.zeros((2, 8), np.float32))
    assert (q == 0).all() and (s == 0).all()
    x = wl.to_bf16_bits(np.array([[1.0, -0.5, 0.25, 127.0]], np.float32))
    q, s = oracle.quantize(x)
    assert q[0].tolist() == [1, 0, 0, 127] and s[0] == 1.0


# ------------------------------------------------------------ weighted variance
def test_weighted_std_integer_weights_closed_form(golden):
    g = golden["weighted_std_integer_weights"]
    eps = 0.125
    y = oracle.weighted_std(np.array(g["x"], np.float32), np.array(g["w"], np.float32), eps=eps)
    mu, var = _frac(g["mean"]), _frac(g["var"])
    np.testing.assert_allclose(y[0], (np.array(g["x"]) - mu) / math.sqrt(var + eps), rtol=1e-14)


def test_weighted_std_is_layernorm_of_the_expanded_row():
    # integer weights: weighted statistics equal those of the repeated multiset
    rng = np.random.default_rng(52)
    x = rng.standard_normal((3, 40)).astype(np.float32)
    w = rng.integers(0, 4, size=40).astype(np.float32)
    w[0] = 1.0
    y = oracle.weighted_std(x, w, eps=1e-3)
    for r in range(3):
        expanded = np.repeat(x[r].astype(np.float64), w.astype(int))
        z = oracle.layernorm(expanded.reshape(1, -1), eps=1e-3)[0]
        # the value at each kept column equals LayerNorm of the expanded row
        firsts = np.cumsum(np.concatenate([[0], w[:-1].astype(int)]))
        keep = w > 0
        np.testing.assert_allclose(y[r, keep], z[firsts[keep]], rtol=1e-12, atol=1e-13)


def test_weighted_std_unit_weights_is_layernorm_and_rejects_bad_weights():
    rng = np.random.default_rng(53)
    x = rng.standard_normal((4, 77)).astype(np.float32)
    np.testing.assert_allclose(oracle.weighted_std(x, np.ones(77, np.float32), eps=1e-5),
                               oracle.layernorm(x, eps=1e-5), rtol=1e-13, atol=1e-13)
    with pytest.raises(ValueError):
        oracle.weighted_std(x, np.zeros(77, np.float32))
    with pytest.raises(ValueError):
        oracle.weighted_std(x, -np.ones(77, np.float32))


# ------------------------------------------------------------------- Pearson
def test_pearson_small_integers_closed_form(golden):
    g = golden["pearson_small_integers"]
    y, r = oracle.pearson(np.array([g["x"]], np.float32), np.array([g["u"]], np.float32))
    den = math.sqrt(_frac(g["var_product"]))
    np.testing.assert_allclose(y[0], [_frac(p) / den for p in g["products"]], rtol=1e-14,
                               atol=1e-15)
    assert r[0] > 0 and abs(r[0] ** 2 - _frac(g["r_squared"])) < 1e-14


def test_pearson_matches_numpy_corrcoef_and_mean_of_outputs():
    # eps = 0: r is the textbook correlation coefficient (numpy's routine),
    # and the row mean of the outputs is r
    rng = np.random.default_rng(61)
    x = rng.standard_normal((5, 300)).astype(np.float32)
    u = (0.7 * x + rng.standard_normal((5, 300))).astype(np.float32)
    y, r = oracle.pearson(x, u)
    for i in range(5):
        ref = np.corrcoef(x[i].astype(np.float64), u[i].astype(np.float64))[0, 1]
        assert abs(r[i] - ref) < 1e-12
        assert abs(y[i].mean() - r[i]) < 1e-12
    assert np.all(np.abs(r) <= 1.0)


def test_pearson_linear_relations_and_symmetry():
    rng = np.random.default_rng(62)
    x = rng.standard_normal((3, 64))
    # u = a x + b: r = +-1 and the outputs are the squared z-scores (times the sign)
    for a, sign in ((4.0, 1.0), (-0.5, -1.0)):
        y, r = oracle.pearson(x, a * x + 3.0)
        np.testing.assert_allclose(r, sign, atol=1e-12)
        z = (x - x.mean(axis=1, keepdims=True)) / x.std(axis=1, keepdims=True)
        np.testing.assert_allclose(y, sign * z * z, rtol=1e-10, atol=1e-12)
    # swapping the operands changes nothing
    u = rng.standard_normal((3, 64))
    y1, r1 = oracle.pearson(x, u)
    y2, r2 = oracle.pearson(u, x)
    np.testing.assert_array_equal(y1, y2)
    np.testing.assert_array_equal(r1, r2)


def test_pearson_eps_closed_form_and_bad_rows():
    # x = u = (1, -1): means 0, variances 1, so y_j = 1 / (1 + eps) = r
    eps = 0.25
    y, r = oracle.pearson(np.array([[1, -1]], np.float32), np.array([[1, -1]], np.float32),
                          eps=eps)
    np.testing.assert_allclose(y[0], [0.8, 0.8], rtol=1e-15)
    np.testing.assert_allclose(r, [0.8], rtol=1e-15)
    # a constant operand with eps = 0 has no correlation; with eps > 0 it gives 0
    c = np.full((1, 8), 3.0, np.float32)
    v = np.arange(8, dtype=np.float32).reshape(1, 8)
    with pytest.raises(ValueError):
        oracle.pearson(c, v)
    y, r = oracle.pearson(c, v, eps=1e-3)
    assert np.all(y == 0.0) and r[0] == 0.0


def test_pearson_bf16_inputs_widen_exactly():
    rng = np.random.default_rng(63)
    x32 = rng.standard_normal((2, 50)).astype(np.float32)
    u32 = rng.standard_normal((2, 50)).astype(np.float32)
    xb, ub = wl.to_bf16_bits(x32), wl.to_bf16_bits(u32)
    y1, r1 = oracle.pearson(xb, ub, eps=1e-5)
    y2, r2 = oracle.pearson(wl.bf16_bits_to_f32(xb), wl.bf16_bits_to_f32(ub), eps=1e-5)
    np.testing.assert_array_equal(y1, y2)
    np.testing.assert_array_equal(r1, r2)
