"""Seeded synthetic inputs for the quantized-KV attention path.

This module is the one place both sides of every parity check draw their
inputs from: the CUDA library (through its Python binding) and the float64
oracle. It holds random number generation, the f32 -> bf16 bit conversion of
generated values, and the shapes of the workloads. It holds none of the
method's arithmetic (no norm, RoPE, quantizer or attention).

Workload shapes follow the e4b layer table of the Gemma 4 pages
(gemma4-e4b.ts, `LAYERS`: sliding layers with a 4- or 8-bit affine cache of
group 64, one full layer in six, KV-shared layers 24..41 reading the last donor
of their own type) and the parity notes of model.ts (full layers: head_dim 512,
one KV head, K = V, partial rotary factor).

Every stream of random numbers is keyed by (seed, purpose, layer, sequence) so
any single sequence of any layer can be regenerated on its own.
"""
from __future__ import annotations

import dataclasses
import numpy as np

GROUP = 64
TILE_KEYS = 64          # cache capacities are kept a multiple of this


# ----------------------------------------------------------------------------
# random streams and bf16 bit patterns of generated values
# ----------------------------------------------------------------------------

def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *key])))


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even of float32 values to bf16 bit patterns (uint16).

    Generated values are finite, so the uint32 sum below cannot wrap."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    u = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return u.astype(np.uint16)


def normal_bf16(seed: int, key: tuple, shape, loc: float = 0.0, scale: float = 1.0) -> np.ndarray:
    """bf16 bit patterns of N(loc, scale^2) draws from the stream `key`."""
    g = _rng(seed, *key)
    a = g.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        a = a * np.float32(scale)
    if loc != 0.0:
        a = a + np.float32(loc)
    return bf16_bits_from_f32(a)


# stream purposes
P_Q, P_K, P_V, P_QW, P_KW, P_CACHE_K, P_CACHE_V, P_BITS, P_LEN, P_ROT = range(10)


# ----------------------------------------------------------------------------
# layer and workload descriptions
# ----------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class LayerSpec:
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    window: int            # 0 = full causal
    rope_dims: int
    rope_theta: float
    k_eq_v: bool
    rms_eps: float = 1e-6
    kv_rotation: bool = False      # the deferred TurboQuant read (rotated K/V, signs from the seed)

    @property
    def group_ratio(self) -> int:
        return self.n_q_heads // self.n_kv_heads


SLIDING = LayerSpec(n_q_heads=8, n_kv_heads=2, head_dim=256, window=512,
                    rope_dims=256, rope_theta=1e4, k_eq_v=False)
FULL_KEQV = LayerSpec(n_q_heads=16, n_kv_heads=1, head_dim=512, window=0,
                      rope_dims=128, rope_theta=1e6, k_eq_v=True)


def round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


def ring_capacity(window: int, rows_per_call: int = 1) -> int:
    """Slots a sliding-window ring needs so that appending `rows_per_call` rows
    never overwrites a key an earlier query of the same call still sees."""
    return round_up(window + rows_per_call - 1, TILE_KEYS)


def linear_capacity(max_pos: int) -> int:
    return round_up(max_pos + 1, TILE_KEYS)


@dataclasses.dataclass
class DecodeWorkload:
    """One decode step of one layer: every sequence has `filled[s]` cached
    tokens (positions 0..filled-1) and appends one token at position filled[s]."""
    name: str
    seed: int
    layer: LayerSpec
    filled: list            # per sequence
    bits: list              # per sequence
    layer_id: int = 0

    @property
    def n_seqs(self) -> int:
        return len(self.filled)

    def capacity(self, s: int) -> int:
        if self.layer.window > 0:
            return ring_capacity(self.layer.window)
        return linear_capacity(self.filled[s])

    def cached_positions(self, s: int) -> np.ndarray:
        """Positions whose rows are still resident before the step's append
        (older rows of a ring were overwritten and are never read)."""
        lo = 0
        if self.layer.window > 0:
            lo = max(0, self.filled[s] - self.capacity(s) + 1)
        return np.arange(lo, self.filled[s], dtype=np.int64)


@dataclasses.dataclass
class PrefillWorkload:
    """One prompt chunk: every sequence holds `filled[s]` cached tokens and
    appends `chunk` new tokens at positions filled[s] .. filled[s]+chunk-1."""
    name: str
    seed: int
    layer: LayerSpec
    filled: list
    chunk: list             # rows per sequence
    bits: list
    layer_id: int = 0

    @property
    def n_seqs(self) -> int:
        return len(self.filled)

    def capacity(self, s: int) -> int:
        if self.layer.window > 0:
            return ring_capacity(self.layer.window, max(self.chunk))
        return linear_capacity(self.filled[s] + self.chunk[s] - 1)

    def cached_positions(self, s: int) -> np.ndarray:
        lo = 0
        if self.layer.window > 0:
            lo = max(0, self.filled[s] - self.capacity(s) + self.chunk[s])
        return np.arange(lo, self.filled[s], dtype=np.int64)


def layer_inputs(seed: int, layer_id: int, layer: LayerSpec, n_rows_q: int, n_rows_kv: int,
                 seq: int | None = None):
    """Norm weights (~1+N(0, 0.1)) and raw q/k/v rows (~N(0,1)) as bf16 bits.

    Returns dict with q [n_rows_q, Hq, D], k [n_rows_kv, Hkv, D], v (or None
    when K = V), q_w [D], k_w [D]."""
    D = layer.head_dim
    sk = () if seq is None else (seq,)
    out = {
        "q_w": normal_bf16(seed, (P_QW, layer_id), (D,), loc=1.0, scale=0.1),
        "k_w": normal_bf16(seed, (P_KW, layer_id), (D,), loc=1.0, scale=0.1),
        "q": normal_bf16(seed, (P_Q, layer_id, *sk), (n_rows_q, layer.n_q_heads, D)),
        "k": normal_bf16(seed, (P_K, layer_id, *sk), (n_rows_kv, layer.n_kv_heads, D)),
        "v": None,
    }
    if not layer.k_eq_v:
        out["v"] = normal_bf16(seed, (P_V, layer_id, *sk), (n_rows_kv, layer.n_kv_heads, D))
    out["rot"] = rotation_signs(seed, layer_id, D) if layer.kv_rotation else None
    return out


def rotation_signs(seed: int, layer_id: int, head_dim: int) -> np.ndarray:
    """int8 [head_dim] of +1 / -1, equally likely: the per-layer signs of the
    rotated (deferred TurboQuant) read."""
    g = _rng(seed, P_ROT, layer_id)
    return np.where(g.random(head_dim) < 0.5, -1, 1).astype(np.int8)


def cache_rows(seed: int, layer_id: int, seq: int, layer: LayerSpec, positions: np.ndarray):
    """Raw k (and v) rows [n, Hkv, D] for the listed cached positions of one
    sequence, as bf16 bits.  The stream is keyed by sequence, so a row's values
    depend only on (seed, layer, sequence, position-index-from-0)."""
    n_all = int(positions[-1]) + 1 if len(positions) else 0
    first = int(positions[0]) if len(positions) else 0
    D, H = layer.head_dim, layer.n_kv_heads
    # Draw only the rows from `first` onward: each stream is generated in
    # fixed blocks of 256 positions so that any suffix can be drawn alone.
    def draw(purpose):
        blocks = []
        b0, b1 = first // 256, (n_all + 255) // 256
        for b in range(b0, b1):
            blocks.append(normal_bf16(seed, (purpose, layer_id, seq, b), (256, H, D)))
        if not blocks:
            return np.zeros((0, H, D), np.uint16)
        a = np.concatenate(blocks, axis=0)
        return a[first - b0 * 256: n_all - b0 * 256]
    k = draw(P_CACHE_K)
    v = None if layer.k_eq_v else draw(P_CACHE_V)
    return k, v


def cache_rows_job(args):
    """cache_rows(*args), for process pools (this module imports no torch)."""
    return cache_rows(*args)


# ----------------------------------------------------------------------------
# the five measured workloads
# ----------------------------------------------------------------------------

def workload_tiny_decode() -> DecodeWorkload:
    """Tiny sliding-window decode: 1 sequence, 8 q / 2 kv heads, head_dim 256,
    128 cached tokens, window 512, 4-bit, full RoPE theta 1e4."""
    return DecodeWorkload("tiny-sliding-decode-b1", 1001, SLIDING, filled=[128], bits=[4])


def workload_sliding_decode_b16() -> DecodeWorkload:
    """Sliding decode, 16 sequences at 4096 cached tokens, window 512;
    sequences 0..7 use a 4-bit cache and 8..15 an 8-bit cache."""
    return DecodeWorkload("sliding-decode-b16-4k-w512", 1002, SLIDING,
                          filled=[4096] * 16, bits=[4] * 8 + [8] * 8)


def workload_full_keqv_decode() -> DecodeWorkload:
    """Full-attention K = V decode: 8 sequences at 32768 cached tokens,
    16 q / 1 kv head, head_dim 512, 128 of 512 dims rotated, theta 1e6, 4-bit."""
    return DecodeWorkload("full-keqv-decode-b8-32k", 1003, FULL_KEQV,
                          filled=[32768] * 8, bits=[4] * 8)


def workload_full_keqv_rotated_decode() -> DecodeWorkload:
    """The full-attention K = V decode above with the deferred TurboQuant read
    (K and V cached in the randomized Hadamard basis, the output rotated back)."""
    base = workload_full_keqv_decode()
    return DecodeWorkload(base.name + "-rotated", base.seed, dataclasses.replace(FULL_KEQV, kv_rotation=True),
                          filled=list(base.filled), bits=list(base.bits))


def workload_prefill_chunk() -> PrefillWorkload:
    """Prompt chunk: 4 sequences append 512 tokens each onto 8192 cached
    tokens of an 8-bit cache; 8 q / 2 kv heads, head_dim 256, window 1024."""
    layer = dataclasses.replace(SLIDING, window=1024)
    return PrefillWorkload("prefill-chunk-b4x512-8k-w1024", 1004, layer,
                           filled=[8192] * 4, chunk=[512] * 4, bits=[8] * 4)


def workload_prefill_full() -> PrefillWorkload:
    """Prompt chunk on a full-attention layer: 4 sequences append 512 tokens
    each onto 8192 cached tokens of a 4-bit cache; 16 q / 1 kv head, head_dim
    512, K = V, partial RoPE on 128 dims."""
    return PrefillWorkload("prefill-full-b4x512-8k-d512", 1009, FULL_KEQV,
                           filled=[8192] * 4, chunk=[512] * 4, bits=[4] * 4)


N_LAYERS = 42
N_DONORS = 24


def stack_layer_kind(i: int) -> str:
    """5 sliding : 1 full, full at layers 5, 11, 17, ... (gemma4-e4b.ts LAYERS)."""
    return "full" if i % 6 == 5 else "sliding"


def stack_cache_layer(i: int) -> int:
    """Index of the layer owning the cache that layer i attends: i itself for
    the donors 0..23; for a sharer, the highest-numbered donor of its own
    attention type (22 when sliding, 23 when full)."""
    if i < N_DONORS:
        return i
    want = stack_layer_kind(i)
    return max(j for j in range(N_DONORS) if stack_layer_kind(j) == want)


@dataclasses.dataclass
class StackWorkload:
    """Decode step over the 42-layer stack for ragged sequences."""
    name: str
    seed: int
    lengths: list          # cached tokens per sequence; new token at this position
    donor_bits: dict       # donor layer -> 4 or 8

    @property
    def n_seqs(self) -> int:
        return len(self.lengths)

    def layer(self, i: int) -> LayerSpec:
        return FULL_KEQV if stack_layer_kind(i) == "full" else SLIDING

    def decode_view(self, i: int) -> DecodeWorkload:
        """The per-layer decode workload of (donor) layer i."""
        d = stack_cache_layer(i)
        return DecodeWorkload(f"{self.name}-layer{d}", self.seed, self.layer(d),
                              filled=list(self.lengths), bits=[self.donor_bits[d]] * self.n_seqs,
                              layer_id=d)


def workload_stack_decode(n_seqs: int = 64, lo: int = 1024, hi: int = 32768) -> StackWorkload:
    """Mixed decode step over the 42-layer stack pattern for ragged sequences
    with lengths uniform in [lo, hi]; per-donor KV bits 4 or 8 from the seed."""
    seed = 1005
    g = _rng(seed, P_LEN)
    lengths = [int(x) for x in g.integers(lo, hi + 1, size=n_seqs)]
    gb = _rng(seed, P_BITS)
    bits = {d: int(gb.choice([4, 8])) for d in range(N_DONORS)}
    return StackWorkload("stack42-mixed-decode-64-ragged", seed, lengths, bits)


# KV bit width of every cache-owning layer 0..23 in the e4b artifact's layer
# table (gemma4-e4b.ts, `LAYERS`); the full-attention donors 5, 11, 17, 23
# are 4, 8, 4, 4 bits, so the full-layer reads of a step are mostly 4-bit
E4B_DONOR_BITS = [4, 4, 4, 8, 8, 4, 4, 4, 4, 8, 8, 8, 4, 4, 8, 4, 4, 4, 4, 4, 4, 4, 4, 4]


def workload_stack_decode_e4b_bits() -> StackWorkload:
    """The 42-layer step of workload_stack_decode with the per-donor bit widths
    of the e4b layer table instead of drawn from the seed."""
    wl = workload_stack_decode()
    return StackWorkload("stack42-e4b-bits-decode-64-ragged", wl.seed, list(wl.lengths),
                         {d: E4B_DONOR_BITS[d] for d in range(N_DONORS)})


def workload_mixed_step(n_decode: int = 48, lo: int = 1024, hi: int = 8192):
    """A mixed step of one sliding layer (the 42-layer stack's sliding shape):
    a decode group of n_decode sequences with lengths uniform in [lo, hi] and
    per-sequence bits from the seed, and a window group of two prompt chunks
    of 256 rows onto 4096 and 6000 cached tokens (8- and 4-bit).  Both groups
    share the seed and layer id, hence the norm weights."""
    seed = 1006
    g = _rng(seed, P_LEN)
    lengths = [int(x) for x in g.integers(lo, hi + 1, size=n_decode)]
    gb = _rng(seed, P_BITS)
    bits = [int(gb.choice([4, 8])) for _ in range(n_decode)]
    dec = DecodeWorkload("mixed-decode-48-ragged", seed, SLIDING, filled=lengths, bits=bits)
    win = PrefillWorkload("mixed-window-2x256", seed, SLIDING, filled=[4096, 6000], chunk=[256, 256],
                          bits=[8, 4])
    return dec, win


def workload_mixed_verify(n_decode: int = 48, n_verify: int = 16, rows: int = 4, lo: int = 1024,
                          hi: int = 8192):
    """A serving step of one sliding layer with speculative verification: a
    decode group of n_decode sequences and a verify group of n_verify other
    sequences, each checking `rows` drafted tokens (a window of `rows` query
    rows); lengths uniform in [lo, hi], per-sequence bits from the seed."""
    seed = 1008
    g = _rng(seed, P_LEN)
    lengths = [int(x) for x in g.integers(lo, hi + 1, size=n_decode + n_verify)]
    gb = _rng(seed, P_BITS)
    bits = [int(gb.choice([4, 8])) for _ in range(n_decode + n_verify)]
    dec = DecodeWorkload(f"verify-decode-{n_decode}-ragged", seed, SLIDING, filled=lengths[:n_decode],
                         bits=bits[:n_decode])
    win = PrefillWorkload(f"verify-window-{n_verify}x{rows}", seed, SLIDING, filled=lengths[n_decode:],
                          chunk=[rows] * n_verify, bits=bits[n_decode:])
    return dec, win


@dataclasses.dataclass
class TrainWorkload:
    """One packed training sequence of a layer under a prefix-shared layout:
    blocks[0] prefix rows (may be 0), blocks[1:] the rows of each branch.  A
    single block is the plain causal training read.  Inputs come from
    `layer_inputs(seed, layer_id, layer, T, T)`."""
    name: str
    seed: int
    layer: LayerSpec
    blocks: list

    @property
    def n_rows(self) -> int:
        return int(sum(self.blocks))

    def offsets(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.blocks)]).astype(np.int32)


def workload_train_prefix_shared(prefix: int = 1024, branches: tuple = (256, 256, 256, 256)):
    """The training forward's read over the 42-layer stack for one packed
    sequence: a prefix of `prefix` rows shared by the given branches (the
    prefix-shared layout of trainable.ts), sliding and full layers of the
    stack's shapes.  Returns (sliding, full) workloads of one seed."""
    seed = 1007
    blocks = [prefix, *branches]
    return (TrainWorkload("train-prefix-sliding", seed, SLIDING, list(blocks)),
            TrainWorkload("train-prefix-full", seed, FULL_KEQV, list(blocks)))


WORKLOADS = {
    "tiny": workload_tiny_decode,
    "sliding16": workload_sliding_decode_b16,
    "full32k": workload_full_keqv_decode,
    "prefill": workload_prefill_chunk,
    "stack42": workload_stack_decode,
}


# ----------------------------------------------------------------------------
# hand-designed rows for the quantizer's edge groups
# ----------------------------------------------------------------------------

# Each entry: name -> {element index: value} of one 64-element group (the rest
# of the group is +0 unless `fill` says otherwise).  The values are exact bf16
# numbers chosen so that the group hits one edge of the affine quantizer.
EDGE_GROUPS = {
    # min -2^-30, max 1, probe 137*2^-12 = half the 4-bit bf16 scale
    # 137*2^-11: the probe sits on a code midpoint only after the fp32
    # subtraction x - min has dropped the 2^-30
    "fp32-quotient-tie-4": ({0: -2.0 ** -30, 1: 1.0, 2: 137 * 2.0 ** -12}, 0.0),
    # the same for 8 bits: bf16 scale 129*2^-15, probe 129*2^-16, min -2^-36
    "fp32-quotient-tie-8": ({0: -2.0 ** -36, 1: 1.0, 2: 129 * 2.0 ** -16}, 0.0),
    # exact half-code values on a scale-1/8 (4-bit) grid
    "ties-grid-4": ({1: 15 / 8, 2: 2.5 / 8, 3: 3.5 / 8, 4: 0.5 / 8, 5: 1.5 / 8, 6: 14.5 / 8}, 0.0),
    # exact half-code values on a scale-1/64 (8-bit) grid
    "ties-grid-8": ({1: 255 / 64, 2: 2.5 / 64, 3: 3.5 / 64, 4: 100.5 / 64, 5: 126.5 / 64}, 0.0),
    # a constant group (scale 0)
    "constant": ({}, 0.5),
    # every zero a -0, so the raw group minimum is -0
    "negative-zero-min": ({1: 1 / 8, 2: 1 / 8, 3: 1 / 8, 4: 1 / 8, 5: 15 / 8}, -0.0),
    # min 0, max 1: the bf16 scale differs from (max - min) / (2^b - 1)
    "bf16-scale-divides": ({1: 1.0, 2: 0.5}, 0.0),
    # a range of one bf16 step above 1
    "nearly-constant": ({63: 1.0078125}, 1.0),
    # an all-negative group
    "all-negative": ({0: -2.0, 1: -0.015625, 2: -1.0, 3: -0.75}, -0.5),
    # a range so small that the scale is a bf16 subnormal: min 0, max 2^-125
    # (4 bits: scale 17 * 2^-133, 8 bits: scale 2^-133); the reciprocal of
    # such a scale overflows float32
    "subnormal-scale": ({1: 2.0 ** -125, 2: 100 * 2.0 ** -133, 3: 37 * 2.0 ** -133}, 0.0),
}

EDGE_HEAD_DIM = 128      # one designed group followed by one balancing group
EDGE_TINY = 2.0 ** -20   # elements below this are left out of the balance


def _bf16_floor(x: float) -> float:
    """The largest bf16 value <= x, for x > 0 (8 significant bits)."""
    m, e = np.frexp(x)                       # x = m * 2^e, m in [0.5, 1)
    return float(np.ldexp(np.floor(np.ldexp(m, 8)), e - 8))


def _balance_group(sum_sq, seed: int) -> np.ndarray:
    """64 bf16 values whose squares sum to exactly `sum_sq` (a Fraction >= 0),
    taken greedily (largest bf16 square that still fits), with seeded signs
    and order.  Raises if 64 values do not suffice."""
    from fractions import Fraction
    rest = Fraction(sum_sq)
    # values are kept on the grid 2^-k with 2^-2k dividing sum_sq, so every
    # remainder stays a whole number of grid squares and the loop ends
    u = rest.denominator.bit_length() - 1          # sum_sq is a multiple of 2^-u
    k = (u + 1) // 2
    grid = 2.0 ** -k
    vals = []
    while rest > 0:
        if len(vals) == GROUP:
            raise ValueError("balancing group needs more than 64 values")
        v = _bf16_floor(float(rest) ** 0.5)
        v = float(np.floor(v / grid)) * grid
        while Fraction(v) ** 2 > rest:          # float sqrt may round up
            v = float(np.floor(_bf16_floor(np.nextafter(v, 0.0)) / grid)) * grid
        vals.append(v)
        rest -= Fraction(v) ** 2
    out = np.zeros(GROUP)
    out[:len(vals)] = vals
    g = _rng(seed, P_CACHE_K, 99)
    out *= np.where(g.random(GROUP) < 0.5, -1.0, 1.0)
    return out[g.permutation(GROUP)]


def quantizer_edge_rows(seed: int = 1007):
    """Rows [n, 1, EDGE_HEAD_DIM] (bf16 bit patterns) whose first group is one
    of EDGE_GROUPS and whose second group makes the squares of the row's
    elements (those of magnitude >= EDGE_TINY) sum to exactly EDGE_HEAD_DIM.
    The row's mean square is then 1 (up to the left-out tiny elements, which
    move it by less than 2^-40 relative), so an RMSNorm without weight and with
    eps 0 leaves every element as it is and the quantizer sees the designed
    group.  Returns (names, bits)."""
    from fractions import Fraction
    names = list(EDGE_GROUPS)
    rows = np.zeros((len(names), 1, EDGE_HEAD_DIM))
    for i, name in enumerate(names):
        at, fill = EDGE_GROUPS[name]
        grp = np.full(GROUP, fill)
        for j, v in at.items():
            grp[j] = v
        big = sum(Fraction(float(v)) ** 2 for v in grp if abs(v) >= EDGE_TINY)
        rows[i, 0, :GROUP] = grp
        rows[i, 0, GROUP:] = _balance_group(Fraction(EDGE_HEAD_DIM) - big, seed + i)
    f32 = rows.astype(np.float32)
    if not np.array_equal(f32.astype(np.float64), rows, equal_nan=False):
        raise ValueError("edge row value not exact in float32")
    bits = bf16_bits_from_f32(f32)
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    if not np.array_equal(back, f32) or not np.array_equal(np.signbit(back), np.signbit(f32)):
        raise ValueError("edge row value not exact in bf16")
    return names, bits
