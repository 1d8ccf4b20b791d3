"""Float64 CPU oracle of attention over a group-wise affine-quantized KV cache.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's CPU
baseline may import this module.  The CUDA library never calls it and shares no
code with it; the two meet only at the seeded inputs of `workloads`.

What is computed, step by step, and where it comes from (the pages are the
three diff pages of the `@mlx-bun/inference` package; cited by file name and
the section of that file):

* q / k RMSNorm per head over head_dim with a learned weight, and an
  un-scaled RMSNorm (no weight) of v -- model.ts, `attentionTraining`
  (`qNorm`, `kNorm`, `vNorm`) and the header's "Parity notes" (on K = V
  layers V comes from the K projection and is normalised without a weight).
* RoPE at the cache position, rotating only `rope_dims` of head_dim (the
  proportional RoPE of model.ts "Parity notes" turns just a
  partial_rotary_factor share of the dims; offset = cache offset,
  `cache.ropePositions` in `attentionTraining`).
* quantize-append of the new K/V rows into a `{bits, groupSize}` affine cache
  (gemma4-e4b.ts, `Gemma4Layer.kv` and the `LAYERS` table: bits 4 or 8, group
  64; the (codes, scales, biases) triple of MLX affine storage, trainable.ts,
  the quantized tied head).  The pages print no quantizer formula; the one
  used is scale = (max - min) / (2^bits - 1), bias = min,
  code = round-half-even((x - bias) / scale) clamped, in IEEE fp32, with codes
  packed little-endian into uint32 words.
* GQA softmax attention with SDPA scale 1.0 (model.ts "Parity notes" and
  `read.attend(q, 1.0)` in `attentionTraining`) under a causal mask, windowed
  on sliding layers (model.ts, `cacheLayers`: a sliding layer's cache is a
  ring sized to its window, and reading it applies the window mask).

Readings taken where the pages are silent:
  R-norm: y = rn_bf16(x / sqrt(mean(x^2) + eps) * w); w = 1 for v.
  R-rope: rotate-half pairs (j, j + R/2) for j < R/2 with frequency
          theta^(-2j/D) over the FULL head_dim D; dims >= R pass through.
          The frequency is taken as its float64 value and the angle is that
          value times the integer position without rounding (positions
          below 2^24).
  R-quant: the stored bf16 scale is the divisor; a constant group has scale
          0 and all codes 0.
  R-window: a query at position p sees keys max(0, p-W+1) .. p (W keys).
  R-round: bf16 rounding after the norm and after RoPE (the pages keep the
          normed and roped tensors as separate bf16 arrays).
  R-zero: a group whose minimum (maximum) is a zero stores +0 as its bias;
          zeros elsewhere keep their IEEE sign.

TurboQuant deferred read of the full-attention caches (model.ts, the
`cacheLayers` comment: the values stay rotated through the fused SDPA and the
read un-rotates the output; `deferredTurboQuantKernels`).  The pages give only
this outline; the rotation is taken from outside them:
  R-rot:  R = diag(s) H, H the Sylvester Hadamard matrix of order head_dim
          (entries +-1, H H^T = D I) and s a vector of +-1 signs drawn once
          per layer (an input, like the norm weights): the randomized Hadamard
          transform, the fast random rotation TurboQuant-style quantizers
          apply before quantizing.  The prepped K and V rows are rotated and
          rounded to bf16 before the quantizer (the same affine groups), q is
          rotated and rounded alike (a zero of a rotated row is +0), the
          scores are (q R)(k R)^T / D = q k^T
          up to those roundings, and the output O' of the rotated values is
          un-rotated: O = O' R^T / D.

The training forward's stateless read (trainable.ts, `trainingCaches` and
`prefixShared.prefixSharedHidden`; model.ts, the `attentionTraining` comment
and `forwardTrainingHidden`): one training cache per donor layer stores
nothing; it reads the plain (unquantized) prepped keys and values handed to it
under the run's mask -- causal (windowed on sliding layers), or block-sparse
with a logical-position window under a prefix-shared layout, whose blocks are
roped block-wise.  A KV-sharing layer reads its donor's keys and values.  The
pages do not print the layout type; the reading taken is
  R-prefix: the packed rows of one training sequence are a prefix block (block
          0, possibly empty) followed by branch blocks 1..n-1, given by block
          offsets.  Prefix row i sits at logical position i, row j of a branch
          at P + j (P = prefix rows).  Row r sees row k iff k is in r's own
          block or in the prefix, lp(k) <= lp(r), and lp(k) > lp(r) - W on a
          sliding layer.  A single block is the plain causal training read.
  Each branch thus reads exactly what it would read as its own sequence
  continuing the prefix.

Values are carried as float64 arrays holding bf16-representable numbers.
"""
from __future__ import annotations

import math
import numpy as np

GROUP = 64


# ----------------------------------------------------------------------------
# bf16 values
# ----------------------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> the float64 values they denote (exact)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """float64 values that are bf16-representable -> their bit patterns."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    if not np.array_equal(f.astype(np.float64), np.asarray(x, dtype=np.float64), equal_nan=True):
        raise ValueError("value not representable in bf16")
    u = f.view(np.uint32)
    if np.any(u & 0xFFFF):
        raise ValueError("value not representable in bf16")
    return (u >> 16).astype(np.uint16)


def rn_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even.

    bf16 keeps 8 significant bits; for |x| in [2^(e-1), 2^e) the spacing is
    2^(e-8), and below the smallest normal (2^-126) the spacing stays 2^-133.
    Magnitudes that round to 2^128 or more become infinities."""
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    e = np.maximum(e, -125)
    q = np.ldexp(np.rint(np.ldexp(x, 8 - e)), e - 8)
    return np.where(np.abs(q) >= 2.0 ** 128, np.copysign(np.inf, x), q)


# ----------------------------------------------------------------------------
# normalisation and rotary embedding
# ----------------------------------------------------------------------------

def rms_norm(x: np.ndarray, w: np.ndarray | None, eps: float) -> np.ndarray:
    """RMSNorm over the last axis (model.ts `attentionTraining`: qNorm / kNorm
    with a weight, vNorm without one), result rounded to bf16."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    y = x / np.sqrt(ms + float(eps))
    if w is not None:
        y = y * np.asarray(w, dtype=np.float64)
    return rn_bf16(y)


def rope_inv_freq(theta: float, head_dim: int, rope_dims: int) -> np.ndarray:
    """theta^(-2j/D) for j < rope_dims/2, the exponent taken over the full
    head_dim (reading R-rope of the "proportional" rotary embedding)."""
    return np.array([math.pow(theta, -(2.0 * j) / head_dim) for j in range(rope_dims // 2)],
                    dtype=np.float64)


def rope_angle(pos: np.ndarray, f: np.ndarray):
    """The angles pos * f [T, half] for integer positions 0 <= pos < 2^24 and
    the float64 frequencies f, as hi + lo equal to the exact product (reading
    R-rope: the frequency is the float64 value of theta^(-2j/D), the angle that
    value times the position, unrounded).  f is split into a 26-bit head and a
    tail (Veltkamp), so pos * head and pos * tail are exact in float64; hi is
    their rounded sum and lo its rounding error (Knuth's two-sum)."""
    p = np.asarray(pos, dtype=np.float64)[:, None]
    if np.any(p < 0) or np.any(p >= 2.0 ** 24) or np.any(p != np.floor(p)):
        raise ValueError("positions must be integers in [0, 2^24)")
    f = np.asarray(f, dtype=np.float64)[None, :]
    t = 134217729.0 * f                       # 2^27 + 1
    head = t - (t - f)
    tail = f - head
    p1, p2 = p * head, p * tail               # both exact
    hi = p1 + p2
    b = hi - p1
    lo = (p1 - (hi - b)) + (p2 - b)
    return hi, lo


def rope(x: np.ndarray, pos: np.ndarray, theta: float, rope_dims: int) -> np.ndarray:
    """Rotary embedding of rows x [..., T, H, D] at positions pos [T].

    Pairs (j, j + R/2), j < R/2, are rotated by angle pos * theta^(-2j/D);
    dims >= R are unchanged.  Result rounded to bf16."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    R = int(rope_dims)
    if R == 0:
        return x.copy()
    half = R // 2
    f = rope_inv_freq(theta, D, R)
    hi, lo = rope_angle(pos, f)                                       # [T, half]
    # cos and sin of hi + lo by the angle-addition formulas
    c = (np.cos(hi) * np.cos(lo) - np.sin(hi) * np.sin(lo))[:, None, :]
    s = (np.sin(hi) * np.cos(lo) + np.cos(hi) * np.sin(lo))[:, None, :]
    y = x.copy()
    x1 = x[..., :half]
    x2 = x[..., half:R]
    y[..., :half] = x1 * c - x2 * s
    y[..., half:R] = x2 * c + x1 * s
    return rn_bf16(y)


def prep_q(q_raw, q_w, pos, theta, rope_dims, eps):
    """q rows [T, Hq, D] -> RoPE(qNorm(q)), as bf16 values."""
    return rope(rms_norm(q_raw, q_w, eps), pos, theta, rope_dims)


def prep_k(k_raw, k_w, pos, theta, rope_dims, eps):
    """k rows [T, Hkv, D] -> RoPE(kNorm(k)), as bf16 values."""
    return rope(rms_norm(k_raw, k_w, eps), pos, theta, rope_dims)


def prep_v(v_raw, eps):
    """v rows [T, Hkv, D] -> vNorm(v) (no weight, no RoPE).  On K = V layers
    the caller passes the raw k rows as v_raw."""
    return rms_norm(v_raw, None, eps)


# ----------------------------------------------------------------------------
# affine group quantization
# ----------------------------------------------------------------------------

def quantize(x: np.ndarray, bits: int):
    """Quantize bf16 rows x [..., D] group-wise (64 elements per group).

    In IEEE fp32:  s32 = (max - min) / (2^bits - 1);  scale = bf16(s32);
    bias = min;  code = clamp(rint((x - bias) / scale), 0, 2^bits - 1),
    rint rounding half to even.  A group with scale 0 gets all codes 0.

    Returns codes uint32 [..., D], scales and biases float64 [..., D/64]
    (bf16 values)."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    if D % GROUP:
        raise ValueError("head_dim must be a multiple of 64")
    g = x.reshape(*x.shape[:-1], D // GROUP, GROUP).astype(np.float32)   # exact
    # a zero minimum / maximum is taken as +0 (reading R-zero: the sign of a
    # zero extremum is otherwise unspecified)
    mn = g.min(axis=-1) + np.float32(0)
    mx = g.max(axis=-1) + np.float32(0)
    levels = np.float32(2 ** bits - 1)
    s32 = (mx - mn) / levels                                     # two fp32 roundings
    s = rn_bf16(s32.astype(np.float64)).astype(np.float32)       # stored bf16 scale
    bias = mn
    safe = np.where(s == 0, np.float32(1), s)
    q = (g - bias[..., None]) / safe[..., None]                  # two fp32 roundings
    c = np.clip(np.rint(q), 0, 2 ** bits - 1)
    c = np.where((s == 0)[..., None], 0, c).astype(np.uint32)
    return (c.reshape(x.shape), s.astype(np.float64), bias.astype(np.float64))


def pack(codes: np.ndarray, bits: int) -> np.ndarray:
    """Pack codes [..., D] little-endian into uint32 words [..., D*bits/32]:
    element e lands in word e*bits//32 at bit offset (e*bits) % 32."""
    per = 32 // bits
    c = np.asarray(codes, dtype=np.uint64)
    D = c.shape[-1]
    c = c.reshape(*c.shape[:-1], D // per, per)
    words = np.zeros(c.shape[:-1], dtype=np.uint64)
    for i in range(per):
        words |= c[..., i] << np.uint64(i * bits)
    return words.astype(np.uint32)


def unpack(words: np.ndarray, bits: int) -> np.ndarray:
    """Inverse of `pack`."""
    per = 32 // bits
    w = np.asarray(words, dtype=np.uint64)
    mask = np.uint64((1 << bits) - 1)
    parts = [(w >> np.uint64(i * bits)) & mask for i in range(per)]
    c = np.stack(parts, axis=-1)
    return c.reshape(*w.shape[:-1], w.shape[-1] * per).astype(np.uint32)


def dequantize(codes: np.ndarray, scales: np.ndarray, biases: np.ndarray) -> np.ndarray:
    """x_hat = code * scale + bias per element, in float64."""
    c = np.asarray(codes, dtype=np.float64)
    D = c.shape[-1]
    c = c.reshape(*c.shape[:-1], D // GROUP, GROUP)
    x = c * np.asarray(scales)[..., None] + np.asarray(biases)[..., None]
    return x.reshape(*x.shape[:-2], D)


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------

def visible_keys(p: int, window: int) -> tuple:
    """Positions a query at position p attends: [max(0, p-W+1), p], or [0, p]
    on a full layer (window 0)."""
    lo = 0 if window <= 0 else max(0, p - window + 1)
    return lo, p


def attend(q_hat: np.ndarray, k_hat: np.ndarray, v_hat: np.ndarray, scale: float = 1.0) -> np.ndarray:
    """Softmax attention of G query heads over n keys of one KV head, scores
    times `scale` (1.0: the SDPA scale of the pages; 1/D on rotated rows).

    q_hat [G, D], k_hat [n, D], v_hat [n, D] -> [G, D], in float64."""
    s = (q_hat @ k_hat.T) * scale                        # [G, n]
    m = s.max(axis=-1, keepdims=True)
    p = np.exp(s - m)
    return (p @ v_hat) / p.sum(axis=-1, keepdims=True)


def attend_cache(q_hat: np.ndarray, p: int, window: int, n_kv_heads: int,
                 k_hat_at, v_hat_at, scale: float = 1.0) -> np.ndarray:
    """Output [Hq, D] of one query token at position p.

    `k_hat_at(lo, hi)` / `v_hat_at(lo, hi)` return dequantized rows
    [hi-lo+1, Hkv, D] for positions lo..hi.  q head h reads kv head
    h // (Hq / Hkv)."""
    Hq, D = q_hat.shape
    G = Hq // n_kv_heads
    lo, hi = visible_keys(p, window)
    K = k_hat_at(lo, hi)
    V = v_hat_at(lo, hi)
    out = np.empty((Hq, D), dtype=np.float64)
    for kvh in range(n_kv_heads):
        out[kvh * G:(kvh + 1) * G] = attend(q_hat[kvh * G:(kvh + 1) * G], K[:, kvh], V[:, kvh], scale)
    return out


# ----------------------------------------------------------------------------
# the rotation of the deferred TurboQuant read (reading R-rot)
# ----------------------------------------------------------------------------

def hadamard(n: int) -> np.ndarray:
    """Sylvester's Hadamard matrix of order n (a power of two): H_1 = [1],
    H_2m = [[H_m, H_m], [H_m, -H_m]]; entries +-1 and H H^T = n I."""
    if n < 1 or n & (n - 1):
        raise ValueError("order must be a power of two")
    H = np.ones((1, 1))
    while H.shape[0] < n:
        H = np.block([[H, H], [H, -H]])
    return H


def rotate(x: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """x R = (x * s) H over the last axis (R = diag(s) H), in float64."""
    s = np.asarray(signs, dtype=np.float64)
    return (np.asarray(x, dtype=np.float64) * s) @ hadamard(s.shape[0])


def unrotate(y: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """y R^T / D = ((y H^T) * s) / D over the last axis, the inverse of rotate."""
    s = np.asarray(signs, dtype=np.float64)
    D = s.shape[0]
    return ((np.asarray(y, dtype=np.float64) @ hadamard(D).T) * s) / D


# ----------------------------------------------------------------------------
# a quantized cache as the oracle models it: one entry per position
# ----------------------------------------------------------------------------

class OracleCache:
    """Quantized K/V history of one sequence of one layer, indexed by position.

    The GPU library stores position j at slot j % capacity; this model keeps
    every position it was given, densely from the lowest one (`base`), so that
    any window can be read back and any ring layout rebuilt from it."""

    def __init__(self, n_kv_heads: int, head_dim: int, bits: int):
        self.H, self.D, self.bits = n_kv_heads, head_dim, bits
        G = head_dim // GROUP
        self.base = 0
        self.kc = np.zeros((0, n_kv_heads, head_dim), np.uint32)
        self.vc = np.zeros((0, n_kv_heads, head_dim), np.uint32)
        self.ks = np.zeros((0, n_kv_heads, G)); self.kb = np.zeros((0, n_kv_heads, G))
        self.vs = np.zeros((0, n_kv_heads, G)); self.vb = np.zeros((0, n_kv_heads, G))
        self.valid = np.zeros(0, bool)

    def _arrays(self):
        return ["kc", "vc", "ks", "kb", "vs", "vb", "valid"]

    def _cover(self, lo, hi):
        """Extend the arrays to hold positions lo .. hi."""
        if len(self.valid) == 0:
            self.base = lo
        if lo < self.base:
            for name in self._arrays():
                a = getattr(self, name)
                z = np.zeros((self.base - lo,) + a.shape[1:], a.dtype)
                setattr(self, name, np.concatenate([z, a]))
            self.base = lo
        n = hi - self.base + 1
        if n > len(self.valid):
            for name in self._arrays():
                a = getattr(self, name)
                z = np.zeros((n - a.shape[0],) + a.shape[1:], a.dtype)
                setattr(self, name, np.concatenate([a, z]))

    def append(self, positions, k_hat, v_hat):
        """Quantize and store prepped rows k_hat / v_hat [T, Hkv, D]."""
        pos = np.asarray(positions, dtype=np.int64)
        if len(pos) == 0:
            return
        self._cover(int(pos.min()), int(pos.max()))
        i = pos - self.base
        kc, ks, kb = quantize(k_hat, self.bits)
        vc, vs, vb = quantize(v_hat, self.bits)
        self.kc[i], self.ks[i], self.kb[i] = kc, ks, kb
        self.vc[i], self.vs[i], self.vb[i] = vc, vs, vb
        self.valid[i] = True

    def _index(self, lo, hi):
        """Array slice of positions lo .. hi, all of which must be cached."""
        a, b = lo - self.base, hi - self.base + 1
        if a < 0 or b > len(self.valid) or not self.valid[a:b].all():
            raise KeyError(f"positions {lo}..{hi} not all cached")
        return slice(a, b)

    def k_hat(self, lo, hi):
        i = self._index(lo, hi)
        return dequantize(self.kc[i], self.ks[i], self.kb[i])

    def v_hat(self, lo, hi):
        i = self._index(lo, hi)
        return dequantize(self.vc[i], self.vs[i], self.vb[i])

    def packed(self, positions):
        """Packed words and bf16 bit patterns of the listed positions:
        (k_words [n, H, D*b/32], k_scales [n, H, D/64], k_biases, v_words,
        v_scales, v_biases)."""
        p = np.asarray(positions, dtype=np.int64) - self.base
        if len(p) and (p.min() < 0 or p.max() >= len(self.valid) or not self.valid[p].all()):
            raise KeyError("position not cached")
        return (pack(self.kc[p], self.bits), f64_to_bf16(self.ks[p]), f64_to_bf16(self.kb[p]),
                pack(self.vc[p], self.bits), f64_to_bf16(self.vs[p]), f64_to_bf16(self.vb[p]))


# ----------------------------------------------------------------------------
# whole steps
# ----------------------------------------------------------------------------

def prep_kv(k_raw, v_raw, k_w, pos, theta, rope_dims, eps):
    """New K/V rows [T, Hkv, D] before quantization: k gets kNorm + RoPE, v gets
    vNorm; with v_raw None (K = V) v is vNorm of the raw k rows."""
    k_hat = prep_k(k_raw, k_w, pos, theta, rope_dims, eps)
    v_hat = prep_v(k_raw if v_raw is None else v_raw, eps)
    return k_hat, v_hat


def rotate_rows(x: np.ndarray, signs) -> np.ndarray:
    """Prepped bf16 rows rotated and rounded to bf16 (reading R-rot); the rows
    themselves when there is no rotation (signs None)."""
    return x if signs is None else rn_bf16(rotate(x, signs) + 0.0)


def finish_read(out: np.ndarray, signs) -> np.ndarray:
    """The read's output: un-rotated when the values were rotated."""
    return out if signs is None else unrotate(out, signs)


def decode_step(layer, cache: OracleCache, p: int, q_raw, q_w, k_raw, v_raw, k_w, signs=None):
    """One decode token of one sequence: append its K/V at position p, then
    attend all q heads.  q_raw [Hq, D], k_raw/v_raw [Hkv, D] (bf16 values);
    signs [D] (+-1) selects the deferred TurboQuant read (None: plain).
    Returns (q_hat [Hq, D], k_hat, v_hat [Hkv, D], out [Hq, D]); on a rotated
    layer q_hat, k_hat and v_hat are the rotated rows."""
    pos = np.array([p])
    k_hat, v_hat = prep_kv(k_raw[None], None if v_raw is None else v_raw[None], k_w, pos,
                           layer.rope_theta, layer.rope_dims, layer.rms_eps)
    k_hat, v_hat = rotate_rows(k_hat, signs), rotate_rows(v_hat, signs)
    cache.append(pos, k_hat, v_hat)
    q_hat = rotate_rows(prep_q(q_raw[None], q_w, pos, layer.rope_theta, layer.rope_dims, layer.rms_eps),
                        signs)[0]
    scale = 1.0 if signs is None else 1.0 / q_hat.shape[-1]
    out = attend_cache(q_hat, p, layer.window, layer.n_kv_heads, cache.k_hat, cache.v_hat, scale)
    return q_hat, k_hat[0], v_hat[0], finish_read(out, signs)


def prefill_chunk(layer, cache: OracleCache, start: int, q_raw, q_w, k_raw, v_raw, k_w,
                  rows=None, signs=None):
    """A chunk of T tokens of one sequence at positions start .. start+T-1:
    append all T K/V rows, then every token attends the keys visible from its
    own position (the chunk's earlier rows included).

    q_raw [T, Hq, D]; `rows` optionally restricts which tokens' outputs are
    computed; signs as for decode_step.  Returns (q_hat [T, Hq, D], k_hat,
    v_hat, {t: out [Hq, D]})."""
    T = q_raw.shape[0]
    pos = np.arange(start, start + T)
    k_hat, v_hat = prep_kv(k_raw, v_raw, k_w, pos, layer.rope_theta, layer.rope_dims,
                           layer.rms_eps)
    k_hat, v_hat = rotate_rows(k_hat, signs), rotate_rows(v_hat, signs)
    cache.append(pos, k_hat, v_hat)
    q_hat = rotate_rows(prep_q(q_raw, q_w, pos, layer.rope_theta, layer.rope_dims, layer.rms_eps), signs)
    scale = 1.0 if signs is None else 1.0 / q_hat.shape[-1]
    outs = {}
    for t in (range(T) if rows is None else rows):
        outs[t] = finish_read(attend_cache(q_hat[t], start + t, layer.window, layer.n_kv_heads,
                                           cache.k_hat, cache.v_hat, scale), signs)
    return q_hat, k_hat, v_hat, outs


# ----------------------------------------------------------------------------
# the training forward's stateless read (reading R-prefix)
# ----------------------------------------------------------------------------

def layout_positions(block_offsets):
    """Block index and logical position of every packed row of a training
    sequence whose blocks are [off[b], off[b+1]): block 0 is the prefix, the
    others are branches continuing it at position P = off[1]."""
    off = np.asarray(block_offsets, dtype=np.int64)
    T = int(off[-1])
    block = np.zeros(T, dtype=np.int64)
    pos = np.zeros(T, dtype=np.int64)
    P = int(off[1]) if len(off) > 1 else 0
    for b in range(len(off) - 1):
        lo, hi = int(off[b]), int(off[b + 1])
        block[lo:hi] = b
        pos[lo:hi] = np.arange(hi - lo) + (0 if b == 0 else P)
    return block, pos


def train_visible(block_offsets, r: int, window: int) -> np.ndarray:
    """Packed indices of the rows that packed row r reads, in increasing order."""
    block, pos = layout_positions(block_offsets)
    same = (block == block[r]) | (block == 0)
    causal = pos <= pos[r]
    inside = pos > pos[r] - window if window > 0 else np.ones_like(causal)
    return np.nonzero(same & causal & inside)[0]


def train_kv(layer, k_raw, v_raw, k_w, block_offsets):
    """A donor layer's plain keys and values for the packed rows [T, Hkv, D]:
    kNorm + RoPE at each row's logical position, vNorm (K = V: of the raw k
    rows); nothing is quantized."""
    _, pos = layout_positions(block_offsets)
    return prep_kv(k_raw, v_raw, k_w, pos, layer.rope_theta, layer.rope_dims, layer.rms_eps)


def train_attend(layer, q_raw, q_w, k_hat, v_hat, block_offsets, rows=None):
    """The stateless read of the training forward: every packed row's q heads
    attend the rows it sees (train_visible) of k_hat / v_hat [T, Hkv, D] with
    SDPA scale 1.0.  q_raw [T, Hq, D]; `rows` optionally restricts which rows'
    outputs are computed.  Returns (q_hat [T, Hq, D], {r: out [Hq, D]})."""
    _, pos = layout_positions(block_offsets)
    q_hat = prep_q(q_raw, q_w, pos, layer.rope_theta, layer.rope_dims, layer.rms_eps)
    Hq = q_hat.shape[1]
    Hkv = k_hat.shape[1]
    G = Hq // Hkv
    outs = {}
    for r in (range(q_hat.shape[0]) if rows is None else rows):
        vis = train_visible(block_offsets, r, layer.window)
        out = np.empty((Hq, q_hat.shape[2]), dtype=np.float64)
        for kvh in range(Hkv):
            out[kvh * G:(kvh + 1) * G] = attend(q_hat[r, kvh * G:(kvh + 1) * G], k_hat[vis, kvh], v_hat[vis, kvh])
        outs[r] = out
    return q_hat, outs
