"""Expected values of the workloads, computed by the float64 oracle from the
seeded inputs of `workloads` (never from anything the GPU produced)."""
from __future__ import annotations

import dataclasses

import numpy as np

import oracle as O
import workloads as W


def oracle_layer(spec: W.LayerSpec) -> W.LayerSpec:
    """The layer as the library sees it: rms_eps is passed as a float32."""
    return dataclasses.replace(spec, rms_eps=float(np.float32(spec.rms_eps)))


def ring_slots(positions, capacity):
    return np.asarray(positions, dtype=np.int64) % capacity


@dataclasses.dataclass
class SeqExpect:
    cache: O.OracleCache
    fill_positions: np.ndarray
    fill_k_hat: np.ndarray
    fill_v_hat: np.ndarray
    resident: np.ndarray          # positions resident in the cache after the step
    q_hat: np.ndarray             # [rows, Hq, D]
    k_hat: np.ndarray             # new rows [rows, Hkv, D]
    v_hat: np.ndarray
    out: dict                     # row -> [Hq, D]


def signs_of(inp):
    """The layer's rotation signs as float64, or None (no rotation)."""
    return None if inp.get("rot") is None else inp["rot"].astype(np.float64)


def _fill(wl, spec, s, bits):
    L = oracle_layer(spec)
    pos = wl.cached_positions(s)
    cache = O.OracleCache(spec.n_kv_heads, spec.head_dim, bits)
    k_raw, v_raw = W.cache_rows(wl.seed, wl.layer_id, s, spec, pos)
    inp = W.layer_inputs(wl.seed, wl.layer_id, spec, 0, 0)
    k_w = O.bf16_to_f64(inp["k_w"])
    if len(pos):
        kh, vh = O.prep_kv(O.bf16_to_f64(k_raw), None if v_raw is None else O.bf16_to_f64(v_raw), k_w,
                           pos, L.rope_theta, L.rope_dims, L.rms_eps)
        kh, vh = O.rotate_rows(kh, signs_of(inp)), O.rotate_rows(vh, signs_of(inp))
        cache.append(pos, kh, vh)
    else:
        kh = vh = np.zeros((0, spec.n_kv_heads, spec.head_dim))
    return L, cache, pos, kh, vh


def expect_decode(wl: W.DecodeWorkload, s: int) -> SeqExpect:
    spec = wl.layer
    L, cache, pos, kh, vh = _fill(wl, spec, s, wl.bits[s])
    inp = W.layer_inputs(wl.seed, wl.layer_id, spec, wl.n_seqs, wl.n_seqs)
    f = O.bf16_to_f64
    p = wl.filled[s]
    q_hat, k_new, v_new, out = O.decode_step(L, cache, p, f(inp["q"][s]), f(inp["q_w"]), f(inp["k"][s]),
                                             None if inp["v"] is None else f(inp["v"][s]), f(inp["k_w"]),
                                             signs=signs_of(inp))
    cap = wl.capacity(s)
    lo = max(0, p - cap + 1)
    return SeqExpect(cache, pos, kh, vh, np.arange(lo, p + 1), q_hat[None], k_new[None], v_new[None], {0: out})


def expect_shared(donor: SeqExpect, wl: W.DecodeWorkload, layer_id: int, s: int):
    """A KV-shared layer of the stack (gemma4-e4b.ts, LAYERS and the decode
    loop: layers 24..41 attend the cache of the last donor of their attention
    type, with no append): its own q inputs of layer `layer_id`, prepped at the
    sequence's position, attend the donor's cache as the donor's step `donor`
    (an expect_decode of the donor's workload `wl`) left it.
    Returns (q_hat [Hq, D], out [Hq, D])."""
    spec = wl.layer
    L = oracle_layer(spec)
    inp = W.layer_inputs(wl.seed, layer_id, spec, wl.n_seqs, wl.n_seqs)
    f = O.bf16_to_f64
    p = wl.filled[s]
    q_hat = O.prep_q(f(inp["q"][s])[None], f(inp["q_w"]), np.array([p]), L.rope_theta, L.rope_dims,
                     L.rms_eps)[0]
    out = O.attend_cache(q_hat, p, L.window, L.n_kv_heads, donor.cache.k_hat, donor.cache.v_hat)
    return q_hat, out


def expect_prefill(wl: W.PrefillWorkload, s: int, rows=None) -> SeqExpect:
    spec = wl.layer
    L, cache, pos, kh, vh = _fill(wl, spec, s, wl.bits[s])
    inp = W.layer_inputs(wl.seed, wl.layer_id, spec, wl.chunk[s], wl.chunk[s], seq=s)
    f = O.bf16_to_f64
    start = wl.filled[s]
    q_hat, k_new, v_new, outs = O.prefill_chunk(L, cache, start, f(inp["q"]), f(inp["q_w"]), f(inp["k"]),
                                                None if inp["v"] is None else f(inp["v"]), f(inp["k_w"]),
                                                rows=rows, signs=signs_of(inp))
    cap = wl.capacity(s)
    newest = start + wl.chunk[s] - 1
    lo = max(0, newest - cap + 1)
    return SeqExpect(cache, pos, kh, vh, np.arange(lo, newest + 1), q_hat, k_new, v_new, outs)


def compare_cache(gpu_rows: dict, cache: O.OracleCache, positions) -> int:
    """Number of mismatching words/scales/biases between the GPU cache rows
    (gathered at the positions' slots) and the oracle's packed rows."""
    kw, ks, kb, vw, vs, vb = cache.packed(positions)
    # oracle arrays are [n, H, ...]; GPU rows are [H, n, ...]
    pairs = [("k_codes", kw), ("k_scales", ks), ("k_biases", kb),
             ("v_codes", vw), ("v_scales", vs), ("v_biases", vb)]
    bad = 0
    for name, want in pairs:
        got = np.swapaxes(gpu_rows[name], 0, 1)
        bad += int(np.count_nonzero(got != want))
    return bad


def attn_errors(got: np.ndarray, want: np.ndarray):
    d = np.abs(np.asarray(got, dtype=np.float64) - want)
    return float(d.max()), float(d.mean())


# the hand-designed quantizer edge rows of `workloads.quantizer_edge_rows`
EDGE_SPEC = W.LayerSpec(n_q_heads=2, n_kv_heads=1, head_dim=W.EDGE_HEAD_DIM, window=0, rope_dims=0,
                        rope_theta=1e4, k_eq_v=False, rms_eps=0.0)
EDGE_BITS = (4, 8)           # one sequence per bit width, the same rows in each


def edge_inputs(seed: int = 1008):
    """(names, k rows, v rows, q rows, weights) as bf16 bit patterns: K rows are
    the designed rows, V rows the same in reverse order, q rows N(0, 1) draws;
    the q and k norm weights are 1."""
    names, k = W.quantizer_edge_rows()
    v = k[::-1].copy()
    q = W.normal_bf16(seed, (W.P_Q, 0), (len(names), EDGE_SPEC.n_q_heads, EDGE_SPEC.head_dim))
    w = np.full(EDGE_SPEC.head_dim, 0x3F80, np.uint16)          # bf16 1.0
    return names, k, v, q, w


def expect_edge(bits: int) -> SeqExpect:
    """The designed rows as one prompt chunk at position 0 of an empty cache
    with `bits`-bit codes; every row attends."""
    names, k, v, q, w = edge_inputs()
    f = O.bf16_to_f64
    cache = O.OracleCache(1, EDGE_SPEC.head_dim, bits)
    q_hat, k_hat, v_hat, outs = O.prefill_chunk(oracle_layer(EDGE_SPEC), cache, 0, f(q), f(w), f(k), f(v), f(w))
    n = len(names)
    empty = np.zeros((0, 1, EDGE_SPEC.head_dim))
    return SeqExpect(cache, np.arange(0), empty, empty, np.arange(n), q_hat, k_hat, v_hat, outs)


def expect_train(wl: W.TrainWorkload, layer_id: int = 0, rows=None, kv=None):
    """The training read of one layer over the packed sequence of `wl`:
    (k_hat, v_hat, q_hat, {row: out [Hq, D]}).  kv = (k_hat, v_hat) of a donor
    makes it a KV-sharing layer's read (no prep of its own)."""
    spec = oracle_layer(wl.layer)
    T = wl.n_rows
    inp = W.layer_inputs(wl.seed, layer_id, wl.layer, T, T)
    f = O.bf16_to_f64
    off = wl.offsets()
    if kv is None:
        kv = O.train_kv(spec, f(inp["k"]), None if inp["v"] is None else f(inp["v"]), f(inp["k_w"]), off)
    q_hat, outs = O.train_attend(spec, f(inp["q"]), f(inp["q_w"]), kv[0], kv[1], off, rows=rows)
    return kv[0], kv[1], q_hat, outs
