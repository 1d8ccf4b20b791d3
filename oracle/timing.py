"""Times the float64 oracle, as it stands, on a bounded sample of a workload.

TEST INFRASTRUCTURE: run only by bench.py (its CPU baseline and its reference
arm), in a fresh process.

    python oracle/timing.py WORKLOAD STEPS WARMUP NSEQ [PROCS]

Builds the oracle's caches for NSEQ sequences of the workload (untimed),
spread over its length distribution, then times STEPS decode steps after
WARMUP untimed ones.  A step is what the GPU step does for those sequences:
for the 42-layer stack, every donor layer appends the new token and attends,
every KV-shared layer attends its donor's cache.  With PROCS > 1 the sampled
sequences are dealt to PROCS single-threaded worker processes (one per host
core) that start their timed steps together; the step time is the slowest
worker's.  Prints one JSON line.
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
        self.signs = None if inp.get("rot") is None else inp["rot"].astype(np.float64)
        if len(pos):
            kh, vh = O.prep_kv(f(k_raw), None if v_raw is None else f(v_raw), f(inp["k_w"]), pos,
                               spec.rope_theta, spec.rope_dims, eps32(spec))
            self.cache.append(pos, O.rotate_rows(kh, self.signs), O.rotate_rows(vh, self.signs))
        self.p = wl.filled[s]
        self.q, self.q_w = f(inp["q"][s]), f(inp["q_w"])
        self.k, self.k_w = f(inp["k"][s]), f(inp["k_w"])
        self.v = None if inp["v"] is None else f(inp["v"][s])

    def decode(self):
        return O.decode_step(self.spec, self.cache, self.p, self.q, self.q_w, self.k, self.v, self.k_w,
                             signs=self.signs)[3]


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


def sample_indices(lengths, n: int) -> list:
    """n sequences spread over the length distribution: sorted by length, the
    middle one of each of n equal slices (their mean length is close to the
    workload's mean)."""
    order = np.argsort(np.asarray(lengths), kind="stable")
    n = min(n, len(order))
    return sorted({int(order[int((i + 0.5) * len(order) / n)]) for i in range(n)})


def build(workload: str, nseq: int, part=None):
    """(steps callable list, tokens per step, sample description).  `part` =
    (i, P) keeps only the i-th of P interleaved shares of the sample."""
    def share(idx):
        return idx if part is None else idx[part[0]::part[1]]
    if workload in ("stack42", "stack42-e4b"):
        wl = W.workload_stack_decode() if workload == "stack42" else W.workload_stack_decode_e4b_bits()
        idx_all = sample_indices(wl.lengths, nseq)
        idx = share(idx_all)
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
        lens = [wl.lengths[s] for s in idx_all]
        return units, len(idx), (f"{len(idx_all)} of {wl.n_seqs} sequences spread over the length distribution "
                                 f"(indices {idx_all}; mean length {np.mean(lens):.0f}, workload mean "
                                 f"{np.mean(wl.lengths):.0f}), all 42 layers")
    if workload in ("tiny", "sliding16", "full32k", "full32k-8bit", "full32k-rot"):
        if workload == "full32k-8bit":
            base = W.workload_full_keqv_decode()
            wl = W.DecodeWorkload(base.name + "-8bit", base.seed, base.layer, base.filled, [8] * base.n_seqs)
        elif workload == "full32k-rot":
            wl = W.workload_full_keqv_rotated_decode()
        else:
            wl = W.WORKLOADS[workload]()
        idx_all = sample_indices(wl.filled, nseq)
        idx = share(idx_all)
        return ([SeqLayer(wl, s) for s in idx], len(idx),
                f"{len(idx_all)} of {wl.n_seqs} sequences (indices {idx_all})")
    if workload in ("prefill", "prefill-full"):
        wl = W.workload_prefill_chunk() if workload == "prefill" else W.workload_prefill_full()
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


def run_steps(units, steps, warmup, barrier=None) -> float:
    """Seconds per timed step (after `warmup` untimed ones)."""
    for _ in range(warmup):
        for u in units:
            u.decode()
    if barrier is not None:
        barrier.wait()
    t0 = time.perf_counter()
    for _ in range(max(1, steps)):
        for u in units:
            u.decode()
    return (time.perf_counter() - t0) / max(1, steps)


def _worker(workload, nseq, part, steps, warmup, barrier, results):
    units, tokens, sample = build(workload, nseq, part)
    results.put((part[0], tokens, sample, run_steps(units, steps, warmup, barrier)))


def cpu_model() -> str:
    try:
        out = os.popen("lscpu 2>/dev/null").read()
        for ln in out.splitlines():
            if ln.startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def main():
    workload, steps, warmup, nseq = sys.argv[1], int(sys.argv[2]), int(sys.argv[3]), int(sys.argv[4])
    procs = int(sys.argv[5]) if len(sys.argv) > 5 else 1
    if procs <= 1:
        units, tokens, sample = build(workload, nseq)
        dt = run_steps(units, steps, warmup)
    else:
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        barrier, results = ctx.Barrier(procs), ctx.Queue()
        ws = [ctx.Process(target=_worker, args=(workload, nseq, (i, procs), steps, warmup, barrier, results))
              for i in range(procs)]
        for w in ws:
            w.start()
        got = [results.get() for _ in ws]
        for w in ws:
            w.join()
        tokens = sum(g[1] for g in got)
        sample = got[0][2]
        dt = max(g[3] for g in got)          # the workers ran their steps side by side
    print(json.dumps({"tokens_per_s": tokens / dt, "ms_per_step": dt * 1e3, "sample": sample,
                      "tokens_per_step": tokens, "procs": procs, "cpu_model": cpu_model()}))


if __name__ == "__main__":
    main()
