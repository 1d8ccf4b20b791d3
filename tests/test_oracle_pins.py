"""Pins of the float64 oracle to facts outside itself.

The pages print no worked example of the quantizer, the norms, RoPE or the
attention read, so the oracle is pinned by hand-worked cases (derivations in
the comments), closed forms, invariants and brute force on tiny inputs.  Each
pin is a function of the oracle module `o`, so `test_oracle_mutants.py` can
run the same pins against copies of the oracle with a planted mistake and
check that some pin fails.
"""
import math
import os

import numpy as np
import pytest

import oracle as O
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------
# bf16 rounding
# ----------------------------------------------------------------------------

def pin_rn_bf16(o):
    # bf16 has 8 significant bits: in [1, 2) the spacing is 2^-7.
    assert o.rn_bf16(np.array([1.0 + 2 ** -8]))[0] == 1.0               # tie -> even (1.0)
    assert o.rn_bf16(np.array([1.0 + 3 * 2 ** -8]))[0] == 1.0 + 2 ** -6  # tie -> even (up)
    assert o.rn_bf16(np.array([1.0 + 2 ** -8 + 2 ** -30]))[0] == 1.0 + 2 ** -7
    assert o.rn_bf16(np.array([-1.0 - 2 ** -8 - 2 ** -30]))[0] == -1.0 - 2 ** -7
    # every float32 whose low 16 bits are zero is a fixed point
    rng = np.random.default_rng(0)
    u = (rng.integers(0, 2 ** 16, 5000).astype(np.uint32) << 16)
    f = u.view(np.float32)
    f = f[np.isfinite(f)].astype(np.float64)
    assert np.array_equal(o.rn_bf16(f), f)
    # agreement with rounding the float32 bit pattern for float32 inputs
    x = rng.standard_normal(20000).astype(np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    b = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16
    ref = b.astype(np.uint32).view(np.float32).astype(np.float64)
    assert np.array_equal(o.rn_bf16(x.astype(np.float64)), ref)
    # the same over random bit patterns of every finite float32, subnormals
    # (bf16 spacing 2^-133 there) and values that round up to infinity
    # included; the largest float32, (2 - 2^-23) * 2^127, rounds to 2^128 = inf
    u = rng.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32)
    u = u[(u & 0x7F800000) != 0x7F800000]
    u = np.concatenate([u, np.array([0x00000001, 0x807FFFFF, 0x00008000, 0x00018000,
                                     0x7F7FFFFF, 0xFF7F8000, 0x7F7F7FFF], dtype=np.uint32)])
    x = u.view(np.float32)
    b = u.astype(np.uint64)
    b = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16
    ref = b.astype(np.uint32).view(np.float32).astype(np.float64)
    got = o.rn_bf16(x.astype(np.float64))
    assert np.array_equal(got, ref)
    assert np.isinf(o.rn_bf16(np.array([3.4028234663852886e38])))[0]
    assert o.rn_bf16(np.array([2.0 ** -140]))[0] == 0.0          # below half of 2^-133
    assert o.rn_bf16(np.array([3 * 2.0 ** -134]))[0] == 2.0 ** -132   # tie -> even


def test_rn_bf16():
    pin_rn_bf16(O)


# ----------------------------------------------------------------------------
# quantizer, hand-worked cases
# ----------------------------------------------------------------------------

def pin_quant_ramp4(o):
    # x_i = (i mod 16) * 0.25: max - min = 3.75, 3.75 / 15 = 0.25 exactly, so
    # scale 0.25, bias 0, codes i mod 16; word 0 holds codes 0..7 low nibble
    # first: 0x76543210.
    x = (np.arange(64) % 16) * 0.25
    c, s, b = o.quantize(x[None], 4)
    assert s[0, 0] == 0.25 and b[0, 0] == 0.0
    assert np.array_equal(c[0], np.arange(64) % 16)
    w = o.pack(c, 4)
    assert w[0, 0] == 0x76543210 and w[0, 1] == 0xFEDCBA98


def pin_quant_exact8(o):
    # x_i = c_i / 64 with integer c_i in [0, 255] including 0 and 255:
    # (255/64) / 255 = 1/64 exactly -> scale 1/64, bias 0, codes c_i.
    rng = np.random.default_rng(1)
    ci = rng.integers(0, 256, 64)
    ci[3], ci[40] = 0, 255
    c, s, b = o.quantize((ci / 64.0)[None], 8)
    assert s[0, 0] == 1 / 64 and b[0, 0] == 0.0
    assert np.array_equal(c[0], ci)
    w = o.pack(np.array([[1, 2, 3, 4]]), 8)
    assert w[0, 0] == 0x04030201


def pin_quant_constant(o):
    # a constant group: max == min -> scale 0, every code 0, bias = the value
    c, s, b = o.quantize(np.full((1, 64), -1.375), 4)
    assert s[0, 0] == 0.0 and b[0, 0] == -1.375 and not c.any()
    assert np.all(o.dequantize(c, s, b) == -1.375)


def pin_quant_negative_zero(o):
    # reading R-zero: a -0 group minimum is stored as +0; the codes are as for +0
    x = np.full(64, -0.0)           # every zero is -0, so the raw minimum is -0
    x[5] = 15.0
    x[1:5] = 1.0
    c, s, b = o.quantize(x[None], 4)
    assert s[0, 0] == 1.0 and b[0, 0] == 0.0 and not np.signbit(b[0, 0])
    assert o.f64_to_bf16(b)[0, 0] == 0x0000
    assert c[0, 0] == 0 and c[0, 1] == 1 and c[0, 5] == 15
    # the norm keeps the sign of a zero input (IEEE division)
    y = o.rms_norm(np.array([[-0.0, 2.0]]), None, 0.0)
    assert np.signbit(y[0, 0]) and y[0, 0] == 0.0


def pin_quant_ties(o):
    # min 0, max 15 -> scale 1.  (x - 0) / 1 = 2.5 -> 2 and 3.5 -> 4 (half to even)
    x = np.zeros(64)
    x[1], x[2], x[3], x[4] = 15.0, 2.5, 3.5, 0.5
    c, s, _ = o.quantize(x[None], 4)
    assert s[0, 0] == 1.0
    assert (c[0, 2], c[0, 3], c[0, 4], c[0, 1]) == (2, 4, 0, 15)


def pin_quant_bf16_scale_divides(o):
    # The stored bf16 scale is the divisor.  8-bit, min 0 max 1:
    # 1/255 = 2^-8 * 1.0039..., i.e. 128.502 units of 2^-15 -> bf16 scale
    # 129 * 2^-15 = 0.003936767578125.  1 / that = 254.0155 -> code 254
    # (not 255), 0.5 / that = 127.0078 -> code 127.
    x = np.zeros(64)
    x[1], x[2] = 1.0, 0.5
    c, s, _ = o.quantize(x[None], 8)
    assert s[0, 0] == 129 * 2.0 ** -15
    assert (c[0, 1], c[0, 2]) == (254, 127)
    # 4-bit: 1/15 = 136.53 units of 2^-11 -> scale 137 * 2^-11; 1 / scale
    # = 14.9489 -> code 15.
    c, s, _ = o.quantize(x[None], 4)
    assert s[0, 0] == 137 * 2.0 ** -11
    assert c[0, 1] == 15 and c[0, 2] == 7      # 0.5 / s = 7.4745 -> 7


def pin_quant_fp32_quotient(o):
    # The quotient (x - bias) / scale is taken in fp32, after an fp32
    # subtraction.  4-bit, min -2^-30, max 1: fl32(1 + 2^-30) = 1 (fp32 keeps
    # 24 bits), 1/15 = 136.53 units of 2^-11 -> scale 137 * 2^-11.  The probe
    # x = 137 * 2^-12 is half a scale; fl32(x + 2^-30) = x (the fp32 spacing
    # at x is 2^-28), so the quotient is exactly 0.5 and rounds to the even
    # code 0, where the exact quotient 0.5 + 2^-30 / scale would give 1.  The
    # maximum gives 1 / scale = 14.95 -> 15; the zeros give ~2^-26 -> 0.
    x = np.zeros(64)
    x[0], x[1], x[2] = -2.0 ** -30, 1.0, 137 * 2.0 ** -12
    c, s, b = o.quantize(x[None], 4)
    assert s[0, 0] == 137 * 2.0 ** -11 and b[0, 0] == -2.0 ** -30
    assert (c[0, 0], c[0, 1], c[0, 2], c[0, 3]) == (0, 15, 0, 0)
    # 8-bit, min -2^-36: scale 129 * 2^-15 as in the bf16-scale case; the
    # probe 129 * 2^-16 is half a scale and 2^-36 is below half the fp32
    # spacing there (2^-32): code 0.  The maximum: 1 / scale = 254.02 -> 254.
    x[0], x[2] = -2.0 ** -36, 129 * 2.0 ** -16
    c, s, b = o.quantize(x[None], 8)
    assert s[0, 0] == 129 * 2.0 ** -15 and b[0, 0] == -2.0 ** -36
    assert (c[0, 0], c[0, 1], c[0, 2]) == (0, 254, 0)


def pin_quant_group_independence(o):
    # groups of 64 along the row are quantized independently
    rng = np.random.default_rng(2)
    x = o.rn_bf16(rng.standard_normal((3, 256)))
    c, s, b = o.quantize(x, 4)
    for g in range(4):
        cg, sg, bg = o.quantize(x[:, 64 * g:64 * (g + 1)], 4)
        assert np.array_equal(c[:, 64 * g:64 * (g + 1)], cg)
        assert np.array_equal(s[:, g], sg[:, 0]) and np.array_equal(b[:, g], bg[:, 0])


@pytest.mark.parametrize("pin", [pin_quant_ramp4, pin_quant_exact8, pin_quant_constant,
                                 pin_quant_ties, pin_quant_negative_zero, pin_quant_bf16_scale_divides,
                                 pin_quant_fp32_quotient, pin_quant_group_independence])
def test_quant_hand_cases(pin):
    pin(O)


def pin_quant_invariants(o, bits):
    """Codes in range; bias = group min; dequant error <= scale/2 except at the
    clamped top code; the chosen code is a nearest code by brute force; pack
    and unpack are inverse."""
    rng = np.random.default_rng(10 + bits)
    x = o.rn_bf16(rng.standard_normal((200, 256)) * rng.uniform(0.01, 10, (200, 1)))
    c, s, b = o.quantize(x, bits)
    top = 2 ** bits - 1
    assert c.min() >= 0 and c.max() <= top
    g = x.reshape(200, 4, 64)
    assert np.array_equal(b, g.min(-1))
    # the scale is within half a bf16 ulp of (max - min) / top
    s_exact = (g.max(-1) - g.min(-1)) / top
    assert np.all(np.abs(s - s_exact) <= s_exact * 2.0 ** -8 * 1.0001)
    xh = o.dequantize(c, s, b).reshape(200, 4, 64)
    err = np.abs(xh - g)
    slack = top * np.abs(s - s_exact)                  # clamp slack at the top code
    cg = c.reshape(200, 4, 64)
    bound = np.where(cg == top, s[..., None] / 2 + slack[..., None], s[..., None] / 2)
    assert np.all(err <= bound * (1 + 1e-6) + 1e-12)
    # brute force: no code reconstructs x more closely (up to fp32 rounding of
    # the quotient)
    codes = np.arange(top + 1)
    recon = codes[None, None, None, :] * s[..., None, None] + b[..., None, None]
    best = np.min(np.abs(recon - g[..., None]), axis=-1)
    assert np.all(err <= best + s[..., None] * 1e-5 + 1e-12)
    assert np.array_equal(o.unpack(o.pack(c, bits), bits), c)


@pytest.mark.parametrize("bits", [4, 8])
def test_quant_invariants(bits):
    pin_quant_invariants(O, bits)


# ----------------------------------------------------------------------------
# RMSNorm
# ----------------------------------------------------------------------------

def pin_rms_hand(o):
    # x = [1, 2], w = 1, eps = 0: mean square 2.5, 1/sqrt(2.5) = 0.632455532...
    # = 161.909 units of 2^-8 -> 162 * 2^-8 = 0.6328125; 2/sqrt(2.5) =
    # 1.264911 = 161.909 units of 2^-7 -> 1.265625.
    y = o.rms_norm(np.array([[1.0, 2.0]]), None, 0.0)
    assert y[0, 0] == 0.6328125 and y[0, 1] == 1.265625
    # the weight multiplies: w = [2, -0.5] -> [1.265625, -0.6328125]
    y = o.rms_norm(np.array([[1.0, 2.0]]), np.array([2.0, -0.5]), 0.0)
    assert y[0, 0] == 1.265625 and y[0, 1] == -0.6328125
    # one rounding, after the weight: w = 65/64.  1/sqrt(2.5) * 65/64 =
    # 0.642338 = 164.44 units of 2^-8 -> 164/256; 2/sqrt(2.5) * 65/64 =
    # 1.284675 = 164.44 units of 2^-7 -> 164/128.  (Rounding before the weight
    # would give 162/256 * 65/64 = 164.53 units -> 165.)
    y = o.rms_norm(np.array([[1.0, 2.0]]), np.array([65 / 64, 65 / 64]), 0.0)
    assert y[0, 0] == 164 / 256 and y[0, 1] == 164 / 128
    # eps enters under the square root: x = [1, 1], eps = 3 -> 1/sqrt(4) = 0.5
    y = o.rms_norm(np.array([[1.0, 1.0]]), None, 3.0)
    assert np.all(y == 0.5)


def pin_rms_invariants(o):
    rng = np.random.default_rng(3)
    x = o.rn_bf16(rng.standard_normal((50, 256)))
    w = o.rn_bf16(1 + 0.1 * rng.standard_normal(256))
    # scale invariance with eps = 0 (powers of two scale exactly)
    assert np.array_equal(o.rms_norm(x * 8.0, w, 0.0), o.rms_norm(x, w, 0.0))
    # a row of +-c gives sign * w
    row = np.where(rng.random(256) < 0.5, -3.0, 3.0)[None]
    assert np.array_equal(o.rms_norm(row, w, 0.0), np.sign(row) * w)
    # the result has mean square ~1 (w = 1) up to bf16 rounding
    y = o.rms_norm(x, None, 1e-6)
    assert np.allclose(np.mean(y * y, -1), 1.0, rtol=1e-2)


def test_rms_norm():
    pin_rms_hand(O)
    pin_rms_invariants(O)


# ----------------------------------------------------------------------------
# RoPE
# ----------------------------------------------------------------------------

def pin_rope_hand(o):
    # D = R = 4, theta 1e4, pos 1: frequencies 1 and 1e4^(-1/2) = 0.01; pairs
    # (0, 2) and (1, 3).  x = [1, 0, 0, 0] -> x0' = cos 1 = 0.540302 = 138.317
    # units of 2^-8 -> 138/256 = 0.5390625; x2' = sin 1 = 0.841471 = 215.417
    # units of 2^-8 -> 215/256 = 0.83984375.
    y = o.rope(np.array([[[1.0, 0, 0, 0]]]), np.array([1]), 1e4, 4)
    assert np.array_equal(y[0, 0], [138 / 256, 0.0, 215 / 256, 0.0])
    # x = [0, 0, 1, 0] -> x0' = -sin 1 -> -0.83984375, x2' = cos 1
    y = o.rope(np.array([[[0, 0, 1.0, 0]]]), np.array([1]), 1e4, 4)
    assert np.array_equal(y[0, 0], [-215 / 256, 0.0, 138 / 256, 0.0])


def _textbook_rope(x, pos, theta):
    """Non-interleaved ("rotate half") RoPE as complex multiplication:
    z_j = x_j + i x_{j+D/2} times exp(i pos theta^(-2j/D))."""
    D = x.shape[-1]
    h = D // 2
    z = x[..., :h] + 1j * x[..., h:]
    ang = np.asarray(pos, float)[:, None] * theta ** (-2.0 * np.arange(h) / D)
    z = z * np.exp(1j * ang)[:, None, :]
    return np.concatenate([z.real, z.imag], axis=-1)


def pin_rope_invariants(o):
    rng = np.random.default_rng(4)
    x = o.rn_bf16(rng.standard_normal((6, 2, 256)))
    pos = np.array([0, 1, 7, 511, 4096, 32768])
    # pos 0 and R = 0 are the identity
    assert np.array_equal(o.rope(x[:1], np.array([0]), 1e4, 256), x[:1])
    assert np.array_equal(o.rope(x, pos, 1e4, 0), x)
    # R = D is textbook RoPE (then rounded to bf16)
    full = o.rope(x, pos, 1e4, 256)
    assert np.array_equal(full, o.rn_bf16(_textbook_rope(x, pos, 1e4)))
    # partial: the first R dims are textbook RoPE over an R-dim vector whose
    # frequencies are those of the full D; dims >= R untouched
    R = 64
    part = o.rope(x, pos, 1e6, R)
    assert np.array_equal(part[..., R:], x[..., R:])
    theta_eff = 1e6 ** (R / 256)         # theta^(-2j/D) == (theta^(R/D))^(-2j/R)
    ref = _textbook_rope(x[..., :R], pos, theta_eff)
    assert np.allclose(part[..., :R], ref, atol=2 ** -6, rtol=2 ** -7)
    # pair norms are preserved up to bf16 rounding
    n0 = x[..., :32] ** 2 + x[..., 32:64] ** 2
    n1 = part[..., :32] ** 2 + part[..., 32:64] ** 2
    assert np.allclose(n0, n1, rtol=2e-2, atol=1e-3)
    # relative position: q(m).k(n) depends on m - n only
    q = x[:1, :1]
    k = x[1:2, :1]
    d1 = np.sum(o.rope(q, [100], 1e4, 256) * o.rope(k, [90], 1e4, 256))
    d2 = np.sum(o.rope(q, [2010], 1e4, 256) * o.rope(k, [2000], 1e4, 256))
    assert abs(d1 - d2) < 0.1


def _mp_bf16(mpmath, v):
    """A high-precision value rounded to the nearest bf16 (8 significant
    bits), in mpmath; refuses values within 1e-9 units of a tie."""
    if v == 0:
        return 0.0
    _, e = mpmath.frexp(v)                    # v = m * 2^e, |m| in [0.5, 1)
    units = mpmath.ldexp(v, 8 - int(e))
    r = mpmath.nint(units)
    assert abs(abs(units - r) - 0.5) > 1e-9, "too close to a bf16 tie"
    return float(mpmath.ldexp(r, int(e) - 8))


# (theta, head_dim, position, pair index j): cos or sin of the angle lies near
# zero, where rounding the product position * frequency to float64 (an error
# up to 2^-29 at these positions) moves the bf16 result by one unit
ROPE_NEAR_ZERO = [(1e4, 256, 11039086, 13), (1e4, 256, 14207257, 8),
                  (1e6, 512, 11311958, 5), (1e6, 512, 10761476, 17)]


def pin_rope_large_positions(o):
    """Unit vectors rotated at positions up to 2^24 - 1 against cos and sin of
    position * f evaluated by mpmath at 200 bits, f the float64 frequency
    theta^(-2j/D), each rounded to bf16."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.prec = 200
    cases = list(ROPE_NEAR_ZERO)
    rng = np.random.default_rng(9)
    for p in [2 ** 24 - 1, 2 ** 23 + 1, int(rng.integers(2 ** 20, 2 ** 24))]:
        cases += [(1e4, 256, p, j) for j in range(0, 128, 7)]
    for theta, D, p, j in cases:
        x = np.zeros((2, 1, D))
        x[0, 0, j] = 1.0             # -> (cos a, sin a) at (j, j + D/2)
        x[1, 0, j + D // 2] = 1.0    # -> (-sin a, cos a)
        y = o.rope(x, np.array([p, p]), theta, D)
        a = mpmath.mpf(p) * mpmath.mpf(math.pow(theta, -(2.0 * j) / D))
        c, s = _mp_bf16(mpmath, mpmath.cos(a)), _mp_bf16(mpmath, mpmath.sin(a))
        assert (y[0, 0, j], y[0, 0, j + D // 2]) == (c, s), (theta, D, p, j)
        assert (y[1, 0, j], y[1, 0, j + D // 2]) == (-s, c), (theta, D, p, j)
    with pytest.raises(ValueError):
        o.rope(np.zeros((1, 1, 64)), np.array([2 ** 24]), 1e4, 64)


def test_rope():
    pin_rope_hand(O)
    pin_rope_invariants(O)
    pin_rope_large_positions(O)


def read_rope_freqs():
    """{(theta, head_dim): [float64 frequencies]} from tests/golden/rope_freqs.txt
    (written by make_rope_freqs.py with mpmath at 200 bits)."""
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "rope_freqs.txt")
    table = {}
    for ln in open(path):
        if ln.startswith("#") or not ln.strip():
            continue
        theta, D, j, v = ln.split()
        table.setdefault((float(theta), int(D)), []).append((int(j), float.fromhex(v)))
    return {k: [v for _, v in sorted(vs)] for k, vs in table.items()}


def test_rope_frequencies_are_the_nearest_doubles():
    """The oracle's float64 frequencies theta^(-2j/D) (platform pow) are the
    doubles nearest to the exact values, for every j of every rotary layout
    the workloads use: an independent evaluation pins the pow both sides
    call."""
    for (theta, D), want in read_rope_freqs().items():
        got = O.rope_inv_freq(theta, D, D)
        assert len(want) == D // 2
        assert [float(x) for x in got] == want, (theta, D)


# ----------------------------------------------------------------------------
# attention read
# ----------------------------------------------------------------------------

def _cache_with(o, k_hat, v_hat, bits=8):
    c = o.OracleCache(k_hat.shape[1], k_hat.shape[2], bits)
    c.append(np.arange(k_hat.shape[0]), k_hat, v_hat)
    return c


def pin_attention(o):
    rng = np.random.default_rng(5)
    n, H, D, Hq = 40, 2, 64, 8
    kh = o.rn_bf16(rng.standard_normal((n, H, D)))
    vh = o.rn_bf16(rng.standard_normal((n, H, D)))
    cache = _cache_with(o, kh, vh)
    q = o.rn_bf16(rng.standard_normal((Hq, D)))

    def run(p, window, qq=q, c=cache):
        return o.attend_cache(qq, p, window, H, c.k_hat, c.v_hat)

    # one visible key (p = 0, or window 1): the output is that key's v_hat
    assert np.allclose(run(0, 0), np.repeat(cache.v_hat(0, 0)[0], Hq // H, axis=0), atol=1e-12)
    assert np.allclose(run(17, 1), np.repeat(cache.v_hat(17, 17)[0], Hq // H, axis=0), atol=1e-12)
    # window >= p + 1 equals full causal
    assert np.allclose(run(30, 31), run(30, 0), atol=1e-14)
    assert np.allclose(run(30, 1000), run(30, 0), atol=1e-14)
    # keys outside the window (and in the future) do not matter
    kh2, vh2 = kh.copy(), vh.copy()
    kh2[:20] += 3.0
    vh2[:20] -= 5.0
    kh2[31:] *= -1
    c2 = _cache_with(o, kh2, vh2)
    assert np.allclose(run(30, 11, c=c2), run(30, 11), atol=1e-14)
    # GQA: q head h reads kv head h // (Hq / Hkv): heads 0-3 see kv head 0
    out = run(25, 0)
    only0 = o.attend(q[:4], cache.k_hat(0, 25)[:, 0], cache.v_hat(0, 25)[:, 0])
    assert np.allclose(out[:4], only0, atol=1e-14)
    # equal q heads give equal outputs
    q3 = q.copy()
    q3[1] = q3[0]
    o3 = run(25, 0, qq=q3)
    assert np.array_equal(o3[0], o3[1])
    # closed form for two keys: out = v1 + sigmoid(s2 - s1) (v2 - v1)
    K = cache.k_hat(10, 11)[:, 1]
    V = cache.v_hat(10, 11)[:, 1]
    s = q[4:] @ K.T
    sig = 1.0 / (1.0 + np.exp(-(s[:, 1] - s[:, 0])))
    closed = V[0][None] + sig[:, None] * (V[1] - V[0])[None]
    assert np.allclose(run(11, 2)[4:], closed, atol=1e-12)
    # equal logits -> the mean of the values
    kk = np.zeros((2, 1, D)); kk[:] = kh[0, 0]
    vv = vh[:2, :1]
    c4 = _cache_with(o, kk, vv)
    r = o.attend_cache(q[:1], 1, 0, 1, c4.k_hat, c4.v_hat)
    assert np.allclose(r[0], c4.v_hat(0, 1)[:, 0].mean(0), atol=1e-12)
    # scale 1.0 and max subtraction: huge logits stay finite and pick the argmax
    big = run(39, 0, qq=q * 64.0)
    assert np.all(np.isfinite(big))
    # the max is taken per query head: q heads 0 and 1 (both on kv head 0) of
    # logits near +2000 and with the opposite sign stay finite, and head 0
    # returns the value of its largest-logit key (the next logit trails by
    # hundreds, so the other weights are below e^-100)
    kd = cache.k_hat(0, 39)[:, 0]
    qa = np.zeros((Hq, D))
    qa[0], qa[1] = 32.0 * kd[7], -32.0 * kd[7]
    r = run(39, 0, qq=qa)
    assert np.all(np.isfinite(r))
    s0 = np.sort(qa[0] @ kd.T)
    assert s0[-1] - s0[-2] > 100
    top = int(np.argmax(qa[0] @ kd.T))
    assert np.allclose(r[0], cache.v_hat(top, top)[0, 0], atol=1e-12)
    # the output is a convex combination of the visible values
    out = run(39, 8)
    vis = cache.v_hat(32, 39)
    for h in range(Hq):
        lo, hi = vis[:, h // 4].min(0), vis[:, h // 4].max(0)
        assert np.all(out[h] >= lo - 1e-12) and np.all(out[h] <= hi + 1e-12)


def test_attention():
    pin_attention(O)


def pin_brute_force_attention(o):
    """Tiny case summed term by term over explicit (key, dim) loops with the
    softmax written as exp(s_j) / sum exp(s_i) without max subtraction."""
    rng = np.random.default_rng(6)
    n, D = 6, 64
    kh = o.rn_bf16(rng.standard_normal((n, 1, D)) * 0.2)
    vh = o.rn_bf16(rng.standard_normal((n, 1, D)))
    cache = _cache_with(o, kh, vh, bits=4)
    q = o.rn_bf16(rng.standard_normal((1, D)) * 0.2)
    K = cache.k_hat(0, n - 1)[:, 0]
    V = cache.v_hat(0, n - 1)[:, 0]
    # K / V dequantized: codes * scale + bias, rebuilt here from unpacked
    # packed words to tie the attention to the packed storage
    words = cache.packed(np.arange(n))
    kc = o.unpack(words[0], 4)[:, 0]
    ks = o.bf16_to_f64(words[1])[:, 0]
    kb = o.bf16_to_f64(words[2])[:, 0]
    Kb = np.array([[kc[j, d] * ks[j, d // 64] + kb[j, d // 64] for d in range(D)] for j in range(n)])
    assert np.array_equal(K, Kb)
    e = [math.exp(sum(q[0, d] * K[j, d] for d in range(D))) for j in range(n)]
    ref = [sum(e[j] * V[j, d] for j in range(n)) / sum(e) for d in range(D)]
    got = o.attend_cache(q, n - 1, 0, 1, cache.k_hat, cache.v_hat)[0]
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_brute_force_attention():
    pin_brute_force_attention(O)


# ----------------------------------------------------------------------------
# whole steps
# ----------------------------------------------------------------------------

def pin_keqv(o):
    """K = V with w_k = 1 and no RoPE: the K and V caches are bit-identical
    (kNorm with unit weight equals the un-scaled vNorm)."""
    rng = np.random.default_rng(7)
    layer = W.LayerSpec(4, 1, 128, 0, 0, 1e6, True)
    k_raw = o.rn_bf16(rng.standard_normal((5, 1, 128)))
    kh, vh = o.prep_kv(k_raw, None, np.ones(128), np.arange(5), 1e6, 0, layer.rms_eps)
    assert np.array_equal(kh, vh)
    c = o.OracleCache(1, 128, 4)
    c.append(np.arange(5), kh, vh)
    w = c.packed(np.arange(5))
    assert all(np.array_equal(w[i], w[i + 3]) for i in range(3))
    # v gets the un-scaled norm even when k carries a weight (hand case of
    # pin_rms_hand: x = [1, 2] -> [0.6328125, 1.265625]; with w = [2, -0.5]
    # the k side is [1.265625, -0.6328125])
    kh1, vh1 = o.prep_kv(np.array([[[1.0, 2.0]]]), None, np.array([2.0, -0.5]),
                         np.array([3]), 1e4, 0, 0.0)
    assert np.array_equal(kh1[0, 0], [1.265625, -0.6328125])
    assert np.array_equal(vh1[0, 0], [0.6328125, 1.265625])
    # with a weight and RoPE the two differ
    kh2, vh2 = o.prep_kv(k_raw, None, 1 + 0.1 * np.ones(128), np.arange(5), 1e6, 64, 1e-6)
    assert not np.array_equal(kh2, vh2)


def pin_prefill_matches_decode(o):
    """A chunk of T tokens gives the same cache and outputs as T decode steps."""
    rng = np.random.default_rng(8)
    layer = W.LayerSpec(4, 2, 64, 5, 64, 1e4, False)
    T = 7
    qr = o.rn_bf16(rng.standard_normal((T, 4, 64)))
    kr = o.rn_bf16(rng.standard_normal((T, 2, 64)))
    vr = o.rn_bf16(rng.standard_normal((T, 2, 64)))
    qw = o.rn_bf16(1 + 0.1 * rng.standard_normal(64))
    kw = o.rn_bf16(1 + 0.1 * rng.standard_normal(64))
    c1 = o.OracleCache(2, 64, 4)
    _, _, _, outs = o.prefill_chunk(layer, c1, 0, qr, qw, kr, vr, kw)
    c2 = o.OracleCache(2, 64, 4)
    for t in range(T):
        _, _, _, out = o.decode_step(layer, c2, t, qr[t], qw, kr[t], vr[t], kw)
        assert np.allclose(out, outs[t], atol=1e-14)
    for a, b in zip(c1.packed(np.arange(T)), c2.packed(np.arange(T))):
        assert np.array_equal(a, b)
    # a second chunk continues at position T: its rows are placed, rotated and
    # masked at T .. 2T-1, as T more decode steps would do
    qr2, kr2, vr2 = qr[::-1].copy(), kr[::-1].copy(), vr[::-1].copy()
    _, _, _, outs2 = o.prefill_chunk(layer, c1, T, qr2, qw, kr2, vr2, kw)
    for t in range(T):
        _, _, _, out = o.decode_step(layer, c2, T + t, qr2[t], qw, kr2[t], vr2[t], kw)
        assert np.allclose(out, outs2[t], atol=1e-14)
    for a, b in zip(c1.packed(np.arange(2 * T)), c2.packed(np.arange(2 * T))):
        assert np.array_equal(a, b)


def test_steps():
    pin_keqv(O)
    pin_prefill_matches_decode(O)


# ----------------------------------------------------------------------------
# the workload structure against the page's layer table
# ----------------------------------------------------------------------------

def test_stack_matches_e4b_layer_table():
    rows = []
    with open(os.path.join(GOLDEN, "e4b_layers.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            rows.append(line.split())
    assert len(rows) == W.N_LAYERS == 42
    for layer, attn, cache, bits, group, keqv in rows:
        i = int(layer)
        assert W.stack_layer_kind(i) == attn
        assert W.stack_cache_layer(i) == int(cache)
        assert int(group) == W.GROUP == 64 and int(bits) in (4, 8)
    assert sum(1 for r in rows if int(r[0]) == int(r[2])) == W.N_DONORS == 24


# ----------------------------------------------------------------------------
# the deferred TurboQuant read: rotation R = diag(s) H (reading R-rot)
# ----------------------------------------------------------------------------

def _signs(D, seed=3):
    return np.where(np.random.default_rng(seed).random(D) < 0.5, -1.0, 1.0)


def pin_hadamard(o):
    """Sylvester's matrix: H H^T = n I exactly, symmetric, and entry (i, j) is
    (-1)^popcount(i & j), the closed form of the construction."""
    for k in range(10):
        n = 2 ** k
        H = o.hadamard(n)
        assert H.shape == (n, n)
        assert np.array_equal(H @ H.T, n * np.eye(n)) and np.array_equal(H, H.T)
    H = o.hadamard(64)
    i, j = np.meshgrid(np.arange(64), np.arange(64), indexing="ij")
    pop = np.vectorize(lambda v: bin(int(v)).count("1"))(i & j)
    assert np.array_equal(H, np.where(pop % 2 == 0, 1.0, -1.0))
    with pytest.raises(ValueError):
        o.hadamard(48)


def pin_rotation(o):
    """rotate against the definition written out as loops (sign flip, then
    sum over i of x_i s_i (-1)^popcount(i & j)) on small integers (exact in
    float64), the exact inverse, and the norm scaled by D."""
    rng = np.random.default_rng(11)
    for D in (8, 64):
        s = _signs(D, D)
        x = rng.integers(-9, 10, size=(3, D)).astype(np.float64)
        want = np.zeros_like(x)
        for r in range(x.shape[0]):
            for j in range(D):
                want[r, j] = sum(x[r, i] * s[i] * (-1.0) ** bin(i & j).count("1") for i in range(D))
        y = o.rotate(x, s)
        assert np.array_equal(y, want)
        assert np.array_equal(o.unrotate(y, s), x)
        assert np.array_equal((y * y).sum(-1), D * (x * x).sum(-1))


def pin_rotated_attention_identity(o):
    """With no rounding, attention over rotated q, K, V with scores / D, then
    un-rotated, is plain attention (R R^T = D I)."""
    rng = np.random.default_rng(12)
    D, n, G = 64, 10, 3
    s = _signs(D)
    q, K, V = rng.standard_normal((G, D)), rng.standard_normal((n, D)), rng.standard_normal((n, D))
    got = o.unrotate(o.attend(o.rotate(q, s), o.rotate(K, s), o.rotate(V, s), 1.0 / D), s)
    assert np.allclose(got, o.attend(q, K, V), atol=1e-12, rtol=0)


def pin_rotated_step(o):
    """A decode step and a prompt chunk on a rotated 8-bit layer: the rows it
    stores are bf16 values whose un-rotation is the plain prepped row within
    bf16 rounding, and the outputs, like the plain layer's, are within the
    quantization error of exact attention over the unquantized plain rows
    (the rotation changes only which values get rounded)."""
    rng = np.random.default_rng(13)
    layer = W.LayerSpec(4, 1, 64, 0, 64, 1e4, False, rms_eps=1e-6)
    D = layer.head_dim
    s = _signs(D, 5)
    n = 40
    kraw = o.rn_bf16(rng.standard_normal((n + 1, 1, D)))
    vraw = o.rn_bf16(rng.standard_normal((n + 1, 1, D)))
    qraw = o.rn_bf16(rng.standard_normal((3, 4, D)))
    w = o.rn_bf16(1 + 0.1 * rng.standard_normal(D))
    pos = np.arange(n + 1)
    prep = lambda x: o.prep_kv(x, None, w, pos[:len(x)], layer.rope_theta, layer.rope_dims, layer.rms_eps)
    K = prep(kraw)[0][:, 0]                                  # plain prepped rows, exact reference
    V = o.prep_v(vraw, layer.rms_eps)[:, 0]
    qh = o.prep_q(qraw, w, np.array([n, 20, 21]), layer.rope_theta, layer.rope_dims, layer.rms_eps)
    for signs in (None, s):
        kh, vh = o.prep_kv(kraw[:n], vraw[:n], w, pos[:n], layer.rope_theta, layer.rope_dims, layer.rms_eps)
        kr, vr = o.rotate_rows(kh, signs), o.rotate_rows(vh, signs)
        c = o.OracleCache(1, D, 8)
        c.append(pos[:n], kr, vr)
        q_hat, k_new, v_new, out = o.decode_step(layer, c, n, qraw[0], w, kraw[n], vraw[n], w, signs=signs)
        for rows in (q_hat, k_new, v_new, kr, vr):
            assert np.array_equal(o.rn_bf16(rows), rows)
        if signs is not None:
            assert np.max(np.abs(o.unrotate(kr, s) - kh)) <= 2.0 ** -8 * np.max(np.abs(kr)) / np.sqrt(D) * 2
        assert np.max(np.abs(out - o.attend(qh[0], K[:n + 1], V[:n + 1]))) < 0.1
        c2 = o.OracleCache(1, D, 8)
        c2.append(pos[:20], kr[:20], vr[:20])
        chunk = o.prefill_chunk(layer, c2, 20, qraw[1:3], w, kraw[20:22], vraw[20:22], w, signs=signs)[3]
        for t, got in chunk.items():
            assert np.max(np.abs(got - o.attend(qh[1 + t], K[:21 + t], V[:21 + t]))) < 0.1


def test_rotation():
    pin_hadamard(O)
    pin_rotation(O)
    pin_rotated_attention_identity(O)
    pin_rotated_step(O)


# ----------------------------------------------------------------------------
# the training forward's stateless read (reading R-prefix)
# ----------------------------------------------------------------------------

def _train_case(rng, D=32, Hq=4, Hkv=2, lens=(13, 9, 1, 6), window=0, keqv=False, rope=16):
    layer = W.LayerSpec(Hq, Hkv, D, window, rope, 1e4, keqv, rms_eps=1e-6)
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T = int(off[-1])
    raw = lambda h: O.rn_bf16(rng.standard_normal((T, h, D)))
    w = O.rn_bf16(1 + 0.1 * rng.standard_normal(D))
    return layer, off, raw(Hq), raw(Hkv), (None if keqv else raw(Hkv)), w


def _own_sequence(o, layer, q, k, v, w, rows):
    """The rows `rows` (packed indices, in order) as a sequence of their own at
    positions 0 .. n-1, read by the inference definitions (visible_keys /
    attend_cache) over unquantized keys and values: (k_hat, v_hat, outs)."""
    pos = np.arange(len(rows))
    k_hat, v_hat = o.prep_kv(k[rows], None if v is None else v[rows], w, pos, layer.rope_theta,
                             layer.rope_dims, layer.rms_eps)
    q_hat = o.prep_q(q[rows], w, pos, layer.rope_theta, layer.rope_dims, layer.rms_eps)
    at = lambda a: (lambda lo, hi: a[lo:hi + 1])
    outs = [o.attend_cache(q_hat[t], t, layer.window, layer.n_kv_heads, at(k_hat), at(v_hat))
            for t in range(len(rows))]
    return k_hat, v_hat, outs


def pin_train_branches_read_as_own_sequences(o):
    """Under a prefix-shared layout every branch reads exactly what it reads as
    its own sequence continuing the prefix, and the prefix what it reads
    alone: the packed mask and positions against the plain causal read of each
    unpacked sequence (full, windowed and K = V layers; an empty branch)."""
    for seed, kw in ((21, {}), (22, dict(window=5)), (23, dict(keqv=True, lens=(7, 12, 0, 3))),
                     (24, dict(lens=(0, 6, 4), window=3))):
        rng = np.random.default_rng(seed)
        layer, off, q, k, v, w = _train_case(rng, **kw)
        k_hat, v_hat = o.train_kv(layer, k, v, w, off)
        _, outs = o.train_attend(layer, q, w, k_hat, v_hat, off)
        prefix = np.arange(off[0], off[1])
        for b in range(len(off) - 1):
            rows = np.arange(off[b], off[b + 1])
            seq = prefix if b == 0 else np.concatenate([prefix, rows])
            kk, vv, want = _own_sequence(o, layer, q, k, v, w, seq)
            mine = np.arange(len(seq)) if b == 0 else np.arange(len(prefix), len(seq))
            assert np.array_equal(k_hat[rows], kk[mine]) and np.array_equal(v_hat[rows], vv[mine])
            for j, r in enumerate(rows):
                assert np.allclose(outs[int(r)], want[mine[j]], rtol=0, atol=1e-12), (seed, b, j)


def pin_train_branch_independence(o):
    """A branch's outputs do not depend on another branch's rows, nor on the
    order in which the branches are packed."""
    rng = np.random.default_rng(25)
    layer, off, q, k, v, w = _train_case(rng, window=6)
    k_hat, v_hat = o.train_kv(layer, k, v, w, off)
    _, base = o.train_attend(layer, q, w, k_hat, v_hat, off)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    for a in (q2, k2, v2):
        a[off[1]:off[2]] = O.rn_bf16(rng.standard_normal(a[off[1]:off[2]].shape))   # branch 1 replaced
    kh2, vh2 = o.train_kv(layer, k2, v2, w, off)
    _, other = o.train_attend(layer, q2, w, kh2, vh2, off)
    for r in list(range(off[0], off[1])) + list(range(off[2], off[-1])):
        assert np.array_equal(base[r], other[r])
    # branches 1 and 3 swapped in the packing
    lens = np.diff(off)
    order = [0, 3, 2, 1]
    perm = np.concatenate([np.arange(off[b], off[b + 1]) for b in order])
    off_p = np.concatenate([[0], np.cumsum(lens[order])])
    khp, vhp = o.train_kv(layer, k[perm], v[perm], w, off_p)
    _, swapped = o.train_attend(layer, q[perm], w, khp, vhp, off_p)
    for new_r, old_r in enumerate(perm):
        assert np.allclose(swapped[new_r], base[int(old_r)], rtol=0, atol=1e-12)


def test_training_read():
    pin_train_branches_read_as_own_sequences(O)
    pin_train_branch_independence(O)
    # hand case: prefix of 2, branches of 1 and 2 rows; row 4 (branch 2, row 1,
    # logical position 3) reads the prefix and its own branch up to itself
    assert list(O.train_visible([0, 2, 3, 5], 4, 0)) == [0, 1, 3, 4]
    assert list(O.train_visible([0, 2, 3, 5], 4, 2)) == [3, 4]
    assert list(O.train_visible([0, 2, 3, 5], 2, 0)) == [0, 1, 2]
    assert list(O.layout_positions([0, 2, 3, 5])[1]) == [0, 1, 2, 2, 3]
