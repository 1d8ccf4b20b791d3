"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check that
the pins of `test_oracle_pins.py` catch every one of them."""
import os
import types

import numpy as np
import pytest

import test_oracle_pins as P

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "oracle", "kvq_oracle.py")

MUTANTS = {
    "rope-sign": ("y[..., :half] = x1 * c - x2 * s", "y[..., :half] = x1 * c + x2 * s"),
    "rope-freq-over-R": ("f = rope_inv_freq(theta, D, R)", "f = rope_inv_freq(theta, R, R)"),
    "rope-interleaved-pairs": ("x1 = x[..., :half]\n    x2 = x[..., half:R]",
                               "x1 = x[..., 0:R:2]\n    x2 = x[..., 1:R:2]"),
    "norm-weight-dropped": ("y = y * np.asarray(w, dtype=np.float64)", "y = y * 1.0"),
    "norm-eps-outside-sqrt": ("np.sqrt(ms + float(eps))", "(np.sqrt(ms) + float(eps))"),
    "norm-no-mean": ("ms = np.mean(x * x, axis=-1, keepdims=True)",
                     "ms = np.sum(x * x, axis=-1, keepdims=True)"),
    "quant-divide-by-fp32-scale": ("safe = np.where(s == 0, np.float32(1), s)",
                                   "safe = np.where(s == 0, np.float32(1), s32)"),
    "quant-round-half-up": ("c = np.clip(np.rint(q), 0, 2 ** bits - 1)",
                            "c = np.clip(np.floor(q + np.float32(0.5)), 0, 2 ** bits - 1)"),
    "quant-levels-2^b": ("levels = np.float32(2 ** bits - 1)", "levels = np.float32(2 ** bits)"),
    "quant-bias-max": ("bias = mn\n", "bias = mx\n"),
    "pack-big-endian": ("words |= c[..., i] << np.uint64(i * bits)",
                        "words |= c[..., per - 1 - i] << np.uint64(i * bits)"),
    "window-off-by-one": ("max(0, p - window + 1)", "max(0, p - window)"),
    "gqa-modulo-mapping": ("out[kvh * G:(kvh + 1) * G] = attend(q_hat[kvh * G:(kvh + 1) * G], K[:, kvh], V[:, kvh], scale)",
                           "out[kvh * G:(kvh + 1) * G] = attend(q_hat[kvh::n_kv_heads], K[:, kvh], V[:, kvh], scale)"),
    "softmax-unnormalised": ("return (p @ v_hat) / p.sum(axis=-1, keepdims=True)", "return (p @ v_hat)"),
    "sdpa-scale-rsqrt-d": ("s = (q_hat @ k_hat.T) * scale", "s = (q_hat @ k_hat.T) * scale / np.sqrt(q_hat.shape[-1])"),
    "dequant-no-bias": ("x = c * np.asarray(scales)[..., None] + np.asarray(biases)[..., None]",
                        "x = c * np.asarray(scales)[..., None]"),
    "v-norm-weighted": ("v_hat = prep_v(k_raw if v_raw is None else v_raw, eps)",
                        "v_hat = rms_norm(k_raw if v_raw is None else v_raw, k_w, eps)"),
    "quant-signed-zero-bias": ("    mn = g.min(axis=-1) + np.float32(0)\n", "    mn = g.min(axis=-1)\n"),
    "norm-double-rounding": ("y = y * np.asarray(w, dtype=np.float64)",
                             "y = rn_bf16(y) * np.asarray(w, dtype=np.float64)"),
    "prefill-positions-from-zero": ("pos = np.arange(start, start + T)", "pos = np.arange(T)"),
    "quant-quotient-in-f64": ("q = (g - bias[..., None]) / safe[..., None]",
                              "q = (g.astype(np.float64) - bias[..., None]) / safe[..., None]"),
    "bf16-no-subnormal-spacing": ("    e = np.maximum(e, -125)\n", "\n"),
    "bf16-no-overflow": ("return np.where(np.abs(q) >= 2.0 ** 128, np.copysign(np.inf, x), q)", "return q"),
    "softmax-max-over-heads": ("m = s.max(axis=-1, keepdims=True)", "m = s.max()"),
    "norm-one-plus-weight": ("y = y * np.asarray(w, dtype=np.float64)",
                             "y = y * (1.0 + np.asarray(w, dtype=np.float64))"),
    "rope-position-plus-one": ("    p = np.asarray(pos, dtype=np.float64)[:, None]\n",
                               "    p = np.asarray(pos, dtype=np.float64)[:, None] + 1\n"),
    "rope-angle-rounded-to-f64": ("hi, lo = rope_angle(pos, f)",
                                  "hi, lo = np.asarray(pos, dtype=np.float64)[:, None] * f[None, :], 0.0"),
    "rope-partial-ignored": ("    R = int(rope_dims)\n", "    R = D if int(rope_dims) else 0\n"),
    "rope-exponent-j-over-D": ("math.pow(theta, -(2.0 * j) / head_dim)", "math.pow(theta, -(1.0 * j) / head_dim)"),
    "query-excludes-itself": ("return lo, p\n", "return lo, max(lo, p - 1)\n"),
    "window-ignores-full-layer": ("lo = 0 if window <= 0 else max(0, p - window + 1)",
                                  "lo = max(0, p - window + 1)"),
    "prefill-not-causal": ("attend_cache(q_hat[t], start + t,", "attend_cache(q_hat[t], start + T - 1,"),
    "decode-q-norm-uses-k-weight": ("prep_q(q_raw[None], q_w, pos,", "prep_q(q_raw[None], k_w, pos,"),
    "keqv-v-from-roped-k": ("v_hat = prep_v(k_raw if v_raw is None else v_raw, eps)",
                            "v_hat = prep_v(k_hat if v_raw is None else v_raw, eps)"),
    "quant-scale-truncated": ("s = rn_bf16(s32.astype(np.float64)).astype(np.float32)",
                              "s = (s32.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)"),
    "dequant-bias-before-scale": ("x = c * np.asarray(scales)[..., None] + np.asarray(biases)[..., None]",
                                  "x = (c + np.asarray(biases)[..., None]) * np.asarray(scales)[..., None]"),
    "norm-over-heads": ("ms = np.mean(x * x, axis=-1, keepdims=True)", "ms = np.mean(x * x, axis=-2, keepdims=True)"),
    "rope-cos-sin-swapped": ("c = (np.cos(hi) * np.cos(lo) - np.sin(hi) * np.sin(lo))[:, None, :]\n"
                             "    s = (np.sin(hi) * np.cos(lo) + np.cos(hi) * np.sin(lo))[:, None, :]",
                             "s = (np.cos(hi) * np.cos(lo) - np.sin(hi) * np.sin(lo))[:, None, :]\n"
                             "    c = (np.sin(hi) * np.cos(lo) + np.cos(hi) * np.sin(lo))[:, None, :]"),
    "rope-angle-error-sign": ("    lo = (p1 - (hi - b)) + (p2 - b)\n", "    lo = -((p1 - (hi - b)) + (p2 - b))\n"),
    "quant-levels-minus-one": ("s32 = (mx - mn) / levels", "s32 = (mx - mn) / (levels - 1)"),
    "unpack-big-endian": ("parts = [(w >> np.uint64(i * bits)) & mask for i in range(per)]",
                          "parts = [(w >> np.uint64((per - 1 - i) * bits)) & mask for i in range(per)]"),
    "attend-values-reversed": ("return (p @ v_hat) / p.sum(axis=-1, keepdims=True)",
                               "return (p @ v_hat[::-1]) / p.sum(axis=-1, keepdims=True)"),
    "decode-attends-before-append": ("    cache.append(pos, k_hat, v_hat)\n    q_hat = rotate_rows(prep_q(q_raw[None], q_w, pos,",
                                     "    q_hat = rotate_rows(prep_q(q_raw[None], q_w, pos,"),
    "prefill-window-grows-in-chunk": ("attend_cache(q_hat[t], start + t, layer.window,",
                                      "attend_cache(q_hat[t], start + t, layer.window + t,"),
    "bf16-7-bits": ("q = np.ldexp(np.rint(np.ldexp(x, 8 - e)), e - 8)",
                    "q = np.ldexp(np.rint(np.ldexp(x, 7 - e)), e - 7)"),
    # the rotation of the deferred TurboQuant read
    "rot-signs-after-hadamard": ("return (np.asarray(x, dtype=np.float64) * s) @ hadamard(s.shape[0])",
                                 "return (np.asarray(x, dtype=np.float64) @ hadamard(s.shape[0])) * s"),
    "rot-no-signs": ("return (np.asarray(x, dtype=np.float64) * s) @ hadamard(s.shape[0])",
                     "return np.asarray(x, dtype=np.float64) @ hadamard(s.shape[0])"),
    "unrot-no-divide": ("return ((np.asarray(y, dtype=np.float64) @ hadamard(D).T) * s) / D",
                        "return (np.asarray(y, dtype=np.float64) @ hadamard(D).T) * s"),
    "unrot-no-signs": ("return ((np.asarray(y, dtype=np.float64) @ hadamard(D).T) * s) / D",
                       "return (np.asarray(y, dtype=np.float64) @ hadamard(D).T) / D"),
    "hadamard-other-block-order": ("H = np.block([[H, H], [H, -H]])", "H = np.block([[H, H], [-H, H]])"),
    "rot-score-scale-missing": ("    scale = 1.0 if signs is None else 1.0 / q_hat.shape[-1]\n    out = attend_cache(",
                                "    scale = 1.0\n    out = attend_cache("),
    "rot-output-not-unrotated": ("return out if signs is None else unrotate(out, signs)", "return out"),
    "rot-rows-not-rounded": ("return x if signs is None else rn_bf16(rotate(x, signs) + 0.0)",
                             "return x if signs is None else rotate(x, signs) + 0.0"),
    "rot-q-not-rotated": ("    q_hat = rotate_rows(prep_q(q_raw[None], q_w, pos, layer.rope_theta, layer.rope_dims, layer.rms_eps),\n"
                          "                        signs)[0]",
                          "    q_hat = prep_q(q_raw[None], q_w, pos, layer.rope_theta, layer.rope_dims, layer.rms_eps)[0]"),
    # the training forward's stateless read (reading R-prefix)
    "train-branch-pos-from-zero": ("pos[lo:hi] = np.arange(hi - lo) + (0 if b == 0 else P)",
                                   "pos[lo:hi] = np.arange(hi - lo)"),
    "train-branch-pos-packed": ("pos[lo:hi] = np.arange(hi - lo) + (0 if b == 0 else P)",
                                "pos[lo:hi] = np.arange(hi - lo) + lo"),
    "train-branches-see-each-other": ("same = (block == block[r]) | (block == 0)",
                                      "same = np.ones_like(block, dtype=bool)"),
    "train-branch-no-prefix": ("same = (block == block[r]) | (block == 0)", "same = block == block[r]"),
    "train-window-on-packed-index": ("inside = pos > pos[r] - window if window > 0",
                                     "inside = np.arange(len(pos)) > r - window if window > 0"),
}

PINS = [
    P.pin_rn_bf16, P.pin_quant_ramp4, P.pin_quant_exact8, P.pin_quant_constant,
    P.pin_quant_ties, P.pin_quant_negative_zero, P.pin_quant_bf16_scale_divides, P.pin_quant_fp32_quotient,
    P.pin_quant_group_independence,
    lambda o: P.pin_quant_invariants(o, 4), lambda o: P.pin_quant_invariants(o, 8),
    P.pin_rms_hand, P.pin_rms_invariants, P.pin_rope_hand, P.pin_rope_invariants, P.pin_rope_large_positions,
    P.pin_attention, P.pin_brute_force_attention, P.pin_keqv, P.pin_prefill_matches_decode,
    P.pin_hadamard, P.pin_rotation, P.pin_rotated_attention_identity, P.pin_rotated_step,
    P.pin_train_branches_read_as_own_sequences, P.pin_train_branch_independence,
]


def _mutant(old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
    m = types.ModuleType("kvq_oracle_mutant")
    exec(compile(src.replace(old, new), "kvq_oracle_mutant", "exec"), m.__dict__)
    return m


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    m = _mutant(*MUTANTS[name])
    caught = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(m)
        except Exception:          # an assertion or a crash both count as caught
            caught.append(getattr(pin, "__name__", "pin"))
    assert caught, f"no pin catches mutant {name}"
