"""CPU check of the division-free rounding the quantization kernels use.

The kernels compute the int8 code round_half_even(fl(x / s)) without an IEEE
division per element: q = x * fl(1 / s), and only when q lies within 2^-14 of
a half-integer b is fl(x / s) placed against b exactly, from the remainder
x - b s (one fused multiply-add on the GPU; exact, so float64 reproduces it
here).  This test restates those steps in numpy float32 arithmetic and checks
them against numpy's IEEE single division on random values and on the
adversarial values fl(b s) and their float neighbours, for scales from 1e-27
to 1e+18 (the reciprocal path) and outside that range (the division path).
"""
import numpy as np

F = np.float32


def _ulp_pow(ab):
    bits = np.array([ab], np.float32).view(np.uint32) & np.uint32(0x7F800000)
    return bits.view(np.float32)[0]


def _code(x, s):
    if s == 0:
        return 0
    inv = F(1.0) / s if (s >= F(2.0 ** -90) and s <= F(2.0 ** 100)) else F(0)
    if inv == 0:
        c = np.rint(F(x / s))
    else:
        q = F(x * inv)
        c = F(np.rint(q))
        d = F(q - c)
        if abs(d) >= F(0.5) - F(2.0 ** -14):
            b = F(c + (F(0.5) if d > 0 else F(-0.5)))
            rho = F(np.float64(x) - np.float64(b) * np.float64(s))  # exact, as the FMA
            away = rho if b > 0 else -rho
            if abs(b) == F(0.5):
                ha, ht = F(2.0 ** -25), F(2.0 ** -26)
            else:
                ha = ht = F(_ulp_pow(abs(b)) * F(2.0 ** -24))
            out = F(0.5) if b > 0 else F(-0.5)
            if away > F(s * ha):
                c = F(b + out)
            elif away < -F(s * ht):
                c = F(b - out)
            else:
                c = F(np.rint(b))
    return int(max(-127, min(127, int(c))))


def _ref(x, s):
    return 0 if s == 0 else int(max(-127, min(127, int(np.rint(F(x / s))))))


def test_division_free_codes_match_ieee_division():
    rng = np.random.default_rng(11)
    n = 0
    for _ in range(300):
        amax = F(abs(rng.standard_normal()) * 10.0 ** rng.uniform(-25, 18) + 1e-30)
        s = F(amax / F(127.0))
        xs = list((rng.uniform(-1, 1, 20) * amax).astype(np.float32))
        for b in rng.choice(np.arange(-127, 128) + 0.5, 12):
            v = F(F(b) * s)
            up = dn = v
            xs.append(v)
            for _ in range(3):
                up = np.nextafter(up, F(np.inf))
                dn = np.nextafter(dn, F(-np.inf))
                xs += [up, dn]
        for x in xs:
            x = F(x)
            assert _code(x, s) == _ref(x, s), (x, s)
            n += 1
    assert n > 25000


def test_ties_round_to_even_and_tiny_scales_divide():
    # s = 1: exact half-integers are ties
    for k in range(-127, 127):
        x = F(k + 0.5)
        assert _code(x, F(1.0)) == _ref(x, F(1.0)) == int(np.rint(x))
    # a scale below 2^-90 takes the division path
    s = F(1e-30)
    for x in (F(3e-30), F(-1.2e-28), F(5e-31)):
        assert _code(x, s) == _ref(x, s)
