"""The hand-designed quantizer edge rows (`workloads.quantizer_edge_rows`) on
the CPU: each row passes the weightless, eps-0 RMSNorm unchanged (so the
quantizer sees the designed group), and the oracle puts each designed group on
the edge it was designed for.  The GPU side of the same rows is in
test_gpu_parity.py."""
import numpy as np

import oracle as O
import workloads as W
from oracle_ref import EDGE_BITS, EDGE_SPEC, edge_inputs, expect_edge


def _bits(x):
    return O.f64_to_bf16(x)


def test_rows_pass_the_norm_unchanged():
    names, k, v, q, w = edge_inputs()
    assert len(names) == len(W.EDGE_GROUPS)
    for bits in EDGE_BITS:
        e = expect_edge(bits)
        # bit patterns, so that the sign of every zero is compared too
        assert np.array_equal(_bits(e.k_hat), k)
        assert np.array_equal(_bits(e.v_hat), v)
    x = O.bf16_to_f64(k)
    for i, name in enumerate(names):
        at, fill = W.EDGE_GROUPS[name]
        grp = x[i, 0, :64]
        for j in range(64):
            want = at.get(j, fill)
            assert grp[j] == want and np.signbit(grp[j]) == np.signbit(want), (name, j)
        big = x[i, 0][np.abs(x[i, 0]) >= W.EDGE_TINY]
        assert np.sum(big * big) == W.EDGE_HEAD_DIM


def _k_codes(bits, name):
    names, *_ = edge_inputs()
    e = expect_edge(bits)
    i = names.index(name)
    return O.unpack(e.cache.packed([i])[0], bits)[0, 0], e.cache.packed([i])


def test_designed_edges_are_hit():
    # fp32 quotient exactly 0.5 at the probe (element 2) -> even code 0
    c, _ = _k_codes(4, "fp32-quotient-tie-4")
    assert (c[0], c[1], c[2]) == (0, 15, 0)
    c, _ = _k_codes(8, "fp32-quotient-tie-8")
    assert (c[0], c[1], c[2]) == (0, 254, 0)
    # half-code values round to even
    c, _ = _k_codes(4, "ties-grid-4")
    assert tuple(c[1:7]) == (15, 2, 4, 0, 2, 14)
    c, _ = _k_codes(8, "ties-grid-8")
    assert tuple(c[1:6]) == (255, 2, 4, 100, 126)
    # constant group: scale 0, codes 0, bias 0.5 (bf16 0x3F00)
    for bits in EDGE_BITS:
        c, p = _k_codes(bits, "constant")
        assert not c[:64].any() and p[1][0, 0, 0] == 0 and p[2][0, 0, 0] == 0x3F00
    # -0 minimum stored as +0
    for bits in EDGE_BITS:
        _, p = _k_codes(bits, "negative-zero-min")
        assert p[2][0, 0, 0] == 0x0000
    # the bf16 scale is the divisor
    c, _ = _k_codes(8, "bf16-scale-divides")
    assert (c[1], c[2]) == (254, 127)
    c, _ = _k_codes(4, "bf16-scale-divides")
    assert (c[1], c[2]) == (15, 7)
    # a bf16-subnormal scale: 17 * 2^-133 at 4 bits, 2^-133 at 8 bits
    c, p = _k_codes(4, "subnormal-scale")
    assert tuple(c[:4]) == (0, 15, 6, 2) and p[1][0, 0, 0] == 0x0011
    c, p = _k_codes(8, "subnormal-scale")
    assert tuple(c[:4]) == (0, 255, 100, 37) and p[1][0, 0, 0] == 0x0001


def test_every_row_attends():
    for bits in EDGE_BITS:
        e = expect_edge(bits)
        assert sorted(e.out) == list(range(len(W.EDGE_GROUPS)))
        assert all(np.all(np.isfinite(o)) for o in e.out.values())
        assert EDGE_SPEC.rms_eps == 0.0
