"""Property checks of the oracle's quantizer over generated bf16 groups
(hypothesis; CPU only).  Groups are drawn as bf16 bit patterns, so tiny and
large magnitudes, negative zeros, repeated values and constant groups all
occur; magnitudes are bounded by 2^64, far above what the weightless RMS norm
of the method can produce (at most sqrt(head_dim) times the norm weight)."""
import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import example, given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

import oracle as O  # noqa: E402


def _bf16_values(bits_list):
    b = np.array(bits_list, dtype=np.uint16)
    return O.bf16_to_f64(b)


# finite bf16 bit patterns with exponent field below 127 + 64 (|x| < 2^64)
finite_bf16 = st.integers(0, 0xFFFF).filter(lambda u: ((u >> 7) & 0xFF) < 127 + 64)
groups = st.lists(finite_bf16, min_size=64, max_size=64)


@settings(max_examples=400, deadline=None, derandomize=True)
@given(groups, st.sampled_from([4, 8]))
def test_quantizer_properties(bits_list, bits):
    x = _bf16_values(bits_list)[None]
    c, s, b = O.quantize(x, bits)
    c, s, b = c[0], float(s[0, 0]), float(b[0, 0])
    top = 2 ** bits - 1
    g = x[0]
    # codes in range; bias is the group minimum (a zero minimum stored as +0)
    assert c.min() >= 0 and c.max() <= top
    assert b == g.min() and not (b == 0 and np.signbit(b))
    # the scale is the bf16 value nearest (max - min) / (2^b - 1), up to the
    # fp32 rounding of the difference and the quotient
    rng = g.max() - g.min()
    if rng == 0:
        assert s == 0 and not c.any()
        return
    # monotone in x; the minimum takes code 0
    order = np.argsort(g, kind="stable")
    assert np.all(np.diff(c[order].astype(np.int64)) >= 0)
    assert c[np.argmin(g)] == 0
    if rng / top < 2.0 ** -126:
        # a range below bf16's normal range: the scale is the nearest bf16
        # subnormal (spacing 2^-133), possibly 0 -- then every code is 0
        assert abs(s - rng / top) <= 2.0 ** -134 * (1 + 2.0 ** -20)
        if s == 0:
            assert not c.any()
        return
    # the scale is the bf16 value nearest (max - min) / (2^b - 1), up to the
    # fp32 rounding of the difference and the quotient
    assert abs(s - rng / top) <= (rng / top) * (2.0 ** -8 + 2.0 ** -22)
    # the maximum takes the top code (or one below it when the bf16 scale
    # rounded up)
    assert c[np.argmax(g)] >= top - (1 if bits == 8 else 0)
    # dequantized error: half a scale, plus the clamp slack at the top code
    err = np.abs(c * s + b - g)
    slack = top * abs(s - rng / top)
    assert np.all(err <= s / 2 * (1 + 2.0 ** -20) + np.where(c == top, slack, 0) + 2.0 ** -60 * abs(b))
    # pack and unpack are inverse
    assert np.array_equal(O.unpack(O.pack(c[None], bits), bits)[0], c)


@settings(max_examples=100, deadline=None, derandomize=True)
@given(st.lists(groups, min_size=2, max_size=4), st.sampled_from([4, 8]))
def test_groups_are_independent(gs, bits):
    x = np.concatenate([_bf16_values(g) for g in gs])[None]
    c, s, b = O.quantize(x, bits)
    for i, g in enumerate(gs):
        ci, si, bi = O.quantize(_bf16_values(g)[None], bits)
        assert np.array_equal(c[0, 64 * i:64 * (i + 1)], ci[0])
        assert s[0, i] == si[0, 0] and b[0, i] == bi[0, 0]


def _bf16_neighbours(r: float):
    """The bf16 values just below and above the bf16 value r (finite, r != 0)."""
    u = int(np.array([r], dtype=np.float32).view(np.uint32)[0]) >> 16
    def val(v):
        return float(np.array([v << 16], dtype=np.uint32).view(np.float32)[0])
    a, b = val(u - 1), val(u + 1)          # one unit of the magnitude, either way
    return (min(a, b), max(a, b))


@settings(max_examples=2000, deadline=None, derandomize=True)
@given(st.floats(min_value=-2.0 ** 100, max_value=2.0 ** 100, allow_nan=False, allow_infinity=False,
                 width=64).filter(lambda v: v == 0 or abs(v) >= 2.0 ** -120))
@example(1.0 + 2.0 ** -8)                 # tie -> 1.0 (even)
@example(1.0 + 3 * 2.0 ** -8)             # tie -> 1 + 2^-6 (even)
@example(-(1.0 + 2.0 ** -8))
@example((1.0 + 2.0 ** -8) * 2.0 ** -119)
@example(1.0 + 2.0 ** -8 + 2.0 ** -52)    # just above a tie
@example(255.5 * 2.0 ** 40)               # tie at the top of a binade -> next binade
def test_rn_bf16_is_nearest_ties_to_even(x):
    """rn_bf16 on arbitrary float64 values (the norm and rotation outputs are
    float64 before their bf16 rounding), checked against the definition: the
    result is a bf16 value, no neighbouring bf16 value is closer (exact
    arithmetic), and a tie goes to the even mantissa."""
    from fractions import Fraction
    r = float(O.rn_bf16(np.array([x]))[0])
    bits = int(np.array([r], dtype=np.float32).view(np.uint32)[0])
    assert float(np.float32(r)) == r and bits & 0xFFFF == 0
    if x == 0:
        assert r == 0
        return
    lo, hi = _bf16_neighbours(r)
    d = abs(Fraction(x) - Fraction(r))
    assert d <= abs(Fraction(x) - Fraction(lo)) and d <= abs(Fraction(x) - Fraction(hi))
    if d == abs(Fraction(x) - Fraction(lo)) or d == abs(Fraction(x) - Fraction(hi)):
        assert (bits >> 16) & 1 == 0, "a tie must round to the even mantissa"


def _mp_round_bf16(mpmath, v):
    """(nearest bf16 of the high-precision value v, distance of v from a bf16
    tie in units of the bf16 spacing)."""
    if v == 0:
        return 0.0, 1.0
    _, e = mpmath.frexp(v)
    e = max(int(e), -125)
    units = mpmath.ldexp(v, 8 - e)
    n = mpmath.nint(units)
    return float(mpmath.ldexp(n, e - 8)), float(abs(abs(units - mpmath.floor(units)) - 0.5))


# bf16 values of magnitude 2^-20 .. 2^8: sign, exponent field and mantissa drawn directly
elem_bf16 = st.tuples(st.integers(0, 1), st.integers(127 - 20, 127 + 7), st.integers(0, 127)).map(
    lambda t: (t[0] << 15) | (t[1] << 7) | t[2])
row_bf16 = st.lists(elem_bf16, min_size=64, max_size=64)
weight_bf16 = st.lists(st.integers(0x3F00, 0x4000), min_size=64, max_size=64)     # 0.5 .. 2


@settings(max_examples=60, deadline=None, derandomize=True)
@given(row_bf16, weight_bf16, st.sampled_from([0.0, 1e-6, 0.5]))
def test_rms_norm_is_the_correctly_rounded_definition(xb, wb, eps):
    """RMSNorm against mpmath at 120 bits: y_i is the bf16 value nearest
    x_i / sqrt(mean(x^2) + eps) * w_i (elements within 2^-40 of a tie aside,
    where the float64 oracle's own rounding could decide)."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.prec = 120
    x, w = _bf16_values(xb), _bf16_values(wb)
    y = O.rms_norm(x[None], w, eps)[0]
    ms = mpmath.fsum(mpmath.mpf(float(v)) ** 2 for v in x) / len(x)
    inv = 1 / mpmath.sqrt(ms + mpmath.mpf(float(np.float64(eps))))
    for i in range(len(x)):
        want, tie_dist = _mp_round_bf16(mpmath, mpmath.mpf(float(x[i])) * inv * mpmath.mpf(float(w[i])))
        if tie_dist > 2.0 ** -40:
            assert y[i] == want, (i, x[i], w[i], y[i], want)


@settings(max_examples=60, deadline=None, derandomize=True)
@given(row_bf16, st.integers(0, 2 ** 24 - 1), st.sampled_from([(1e4, 64), (1e6, 32)]))
def test_rope_is_the_correctly_rounded_definition(xb, pos, theta_r):
    """RoPE against mpmath at 200 bits on general vectors (head_dim 64): each
    rotated element is the bf16 value nearest x_j cos(a) -/+ x_{j+R/2} sin(a),
    a = pos * float64(theta^(-2j/64)); dims >= R unchanged."""
    import math
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.prec = 200
    theta, R = theta_r
    x = _bf16_values(xb)
    y = O.rope(x[None, None], np.array([pos]), theta, R)[0, 0]
    half = R // 2
    assert np.array_equal(y[R:], x[R:])
    for j in range(half):
        a = mpmath.mpf(pos) * mpmath.mpf(math.pow(theta, -(2.0 * j) / 64))
        c, s = mpmath.cos(a), mpmath.sin(a)
        x1, x2 = mpmath.mpf(float(x[j])), mpmath.mpf(float(x[j + half]))
        for idx, v in ((j, x1 * c - x2 * s), (j + half, x2 * c + x1 * s)):
            want, tie_dist = _mp_round_bf16(mpmath, v)
            if tie_dist > 2.0 ** -40:
                assert y[idx] == want, (pos, j, idx, y[idx], want)
