"""Times the float64 oracle, as it stands, on a bounded sample of a workload.

TEST INFRASTRUCTURE: run only by bench.py (its CPU baseline and its reference
arm), in a fresh single-threaded process.

    python oracle/timing.py WORKLOAD STEPS WARMUP NSEQ

Builds the oracle's caches for NSEQ seeded-sampled sequences of the workload
(untimed), then times STEPS decode steps after WARMUP untimed ones.  A step is
what the GPU step does for those sequences: for the 42-layer stack, every
donor layer appends the new token and attends, every KV-shared layer attends
its donor's cache.  Prints one JSON line.
"""
from __future__ import annotations

import json
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402
from oracle import kvq_oracle as O  # noqa: E402


def f(bits):
    return O.bf16_to_f64(bits)


def eps32(spec):
    return float(np.float32(spec.rms_eps))


class SeqLayer:
    """Oracle state of one sampled sequence in one (donor) layer."""

    def __init__(self, wl, s):
        spec = wl.layer
        self.spec, self.s = spec, s
        self.cache = O.OracleCache(spec.n_kv_heads, spec.head_dim, wl.bits[s])
        pos = wl.cached_positions(s)
        k_raw, v_raw = W.cache_rows(wl.seed, wl.layer_id, s, spec, pos)
        inp = W.layer_inputs(wl.seed, wl.layer_id, spec, wl.n_seqs, wl.n_seqs)
        if len(pos):
            kh, vh = O.prep_kv(f(k_raw), None if v_raw is None else f(v_raw), f(inp["k_w"]), pos,
                               spec.rope_theta, spec.rope_dims, eps32(spec))
            self.cache.append(pos, kh, vh)
        self.p = wl.filled[s]
        self.q, self.q_w = f(inp["q"][s]), f(inp["q_w"])
        self.k, self.k_w = f(inp["k"][s]), f(inp["k_w"])
        self.v = None if inp["v"] is None else f(inp["v"][s])

    def decode(self):
        return O.decode_step(self.spec, self.cache, self.p, self.q, self.q_w, self.k, self.v, self.k_w)[3]


class Sharer:
    """A KV-shared layer: its own q, the donor's cache, no append."""

    def __init__(self, wl_i, s, donor: SeqLayer):
        spec = wl_i.layer
        inp = W.layer_inputs(wl_i.seed, wl_i.layer_id, spec, wl_i.n_seqs, wl_i.n_seqs)
        self.spec, self.donor, self.p = spec, donor, wl_i.filled[s]
        self.q, self.q_w = f(inp["q"][s]), f(inp["q_w"])

    def decode(self):
        spec = self.spec
        q_hat = O.prep_q(self.q[None], self.q_w, np.array([self.p]), spec.rope_theta, spec.rope_dims,
                         eps32(spec))[0]
        c = self.donor.cache
        return O.attend_cache(q_hat, self.p, spec.window, spec.n_kv_heads, c.k_hat, c.v_hat)


def build(workload: str, nseq: int):
    """(steps callable list, tokens per step, sample description)."""
    if workload == "stack42":
        wl = W.workload_stack_decode()
        idx = sorted(np.random.default_rng(7).choice(wl.n_seqs, size=nseq, replace=False).tolist())
        units = []
        donors = {}
        for i in range(W.N_LAYERS):
            d = W.stack_cache_layer(i)
            for s in idx:
                if i < W.N_DONORS:
                    sl = SeqLayer(wl.decode_view(i), s)
                    donors[(i, s)] = sl
                    units.append(sl)
                else:
                    v = wl.decode_view(i)
                    vi = W.DecodeWorkload(v.name, wl.seed, v.layer, v.filled, v.bits, layer_id=i)
                    units.append(Sharer(vi, s, donors[(d, s)]))
        lens = [wl.lengths[s] for s in idx]
        return units, len(idx), f"{len(idx)} of {wl.n_seqs} sequences (indices {idx}, lengths {lens}), all 42 layers"
    if workload in ("tiny", "sliding16", "full32k"):
        wl = W.WORKLOADS[workload]()
        n = min(nseq, wl.n_seqs)
        idx = sorted(np.random.default_rng(7).choice(wl.n_seqs, size=n, replace=False).tolist())
        return [SeqLayer(wl, s) for s in idx], n, f"{n} of {wl.n_seqs} sequences (indices {idx})"
    if workload == "prefill":
        wl = W.workload_prefill_chunk()
        s = 0
        spec = wl.layer
        rows = 32
        state = SeqLayer(W.DecodeWorkload(wl.name, wl.seed, spec, wl.filled, wl.bits), s)
        inp = W.layer_inputs(wl.seed, wl.layer_id, spec, wl.chunk[s], wl.chunk[s], seq=s)

        class Chunk:
            def decode(self_inner):
                return O.prefill_chunk(spec, state.cache, wl.filled[s], f(inp["q"]), f(inp["q_w"]), f(inp["k"]),
                                       None if inp["v"] is None else f(inp["v"]), f(inp["k_w"]),
                                       rows=range(rows))[3]
        return [Chunk()], rows, f"sequence 0: its whole chunk appended, attention of its first {rows} rows"
    if workload == "mixed":
        dwl, pwl = W.workload_mixed_step()
        n = min(nseq, dwl.n_seqs)
        idx = sorted(np.random.default_rng(7).choice(dwl.n_seqs, size=n, replace=False).tolist())
        units = [SeqLayer(dwl, s) for s in idx]
        s, spec, rows = 0, pwl.layer, 16
        state = SeqLayer(W.DecodeWorkload(pwl.name, pwl.seed, spec, pwl.filled, pwl.bits), s)
        inp = W.layer_inputs(pwl.seed, pwl.layer_id, spec, pwl.chunk[s], pwl.chunk[s], seq=s)

        class WindowRows:
            def decode(self_inner):
                return O.prefill_chunk(spec, state.cache, pwl.filled[s], f(inp["q"]), f(inp["q_w"]), f(inp["k"]),
                                       None if inp["v"] is None else f(inp["v"]), f(inp["k_w"]),
                                       rows=range(rows))[3]
        units.append(WindowRows())
        return units, n + rows, (f"decode group: {n} of {dwl.n_seqs} sequences (indices {idx}); window group: "
                                 f"sequence 0, its chunk appended, attention of its first {rows} rows")
    raise SystemExit(f"unknown workload {workload}")


def main():
    workload, steps, warmup, nseq = sys.argv[1], int(sys.argv[2]), int(sys.argv[3]), int(sys.argv[4])
    units, tokens, sample = build(workload, nseq)
    for _ in range(warmup):
        for u in units:
            u.decode()
    t0 = time.perf_counter()
    for _ in range(max(1, steps)):
        for u in units:
            u.decode()
    dt = (time.perf_counter() - t0) / max(1, steps)
    print(json.dumps({"tokens_per_s": tokens / dt, "ms_per_step": dt * 1e3, "sample": sample,
                      "tokens_per_step": tokens}))


if __name__ == "__main__":
    main()
