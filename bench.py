"""Benchmark of the quantized-KV attention path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step = one pass of the whole hot path over one batch of synthetic input.
The default workload is the 42-layer mixed decode step: 64 ragged sequences
(lengths uniform in [1024, 32768]), the 5 sliding : 1 full layer pattern of
the e4b layer table, per-donor 4/8-bit caches, KV-shared layers 24..41.  Per
step: 24 quantize-appends (q/k/v prep, quantize, pack) and 42 attention reads
(split-K decode, combine), 64 decode tokens.  Other workloads (--workload):
stack42-e4b, tiny, sliding16, full32k (and its 8-bit and rotated forms),
prefill, prefill-full (a head_dim-512 prompt chunk, row path), mixed,
mixed-verify, train42.

The timed region replays a CUDA graph holding K steps (inputs resident in
HBM); `e2e` repeats K steps through the Python binding with inputs copied
from pinned host memory and outputs copied back every step.  The reference
arm (--impl reference) times the float64 CPU oracle on a bounded sample.
Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def rb_pair(D: int, bits: int) -> int:
    """Bytes of one cached key+value row: packed codes plus bf16 scale and
    bias per 64-group, for K and for V."""
    return 2 * (D * bits // 8 + (D // 64) * 4)


def visible_keys(p: int, window: int) -> int:
    return p + 1 if window <= 0 else min(p + 1, window)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            mp = json.load(f)
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS, "source": "fallback"}

    def find(d, keys):
        if isinstance(d, dict):
            for k, v in d.items():
                if k in keys and isinstance(v, (int, float)):
                    return float(v)
                r = find(v, keys)
                if r is not None:
                    return r
        return None
    hbm = find(mp, {"hbm_gbs", "hbm_GBps", "hbm_copy_gbs"})
    # the burst figure: every timed kernel here runs inside a sub-millisecond
    # step, not a seconds-long loop at the power cap
    bf = find(mp, {"bf16_tflops"}) or find(mp, {"bf16_tflops_sustained"})
    return {"hbm_gbs": hbm or FALLBACK_HBM_GBS, "bf16_tflops": bf or FALLBACK_BF16_TFLOPS,
            "source": "measured" if hbm else "fallback"}


# The sources that make up one kernel: its translation unit and every header
# of this repository it includes (the launch plan and the launch live in the
# same .cu).  A traffic figure stays valid while these files are unchanged.
KERNEL_SOURCES = {
    "decode_kernel_512": ["quantized_kv_attention_quant_gb300/csrc/kvq_decode.cu",
                          "quantized_kv_attention_quant_gb300/csrc/kvq_common.cuh",
                          "quantized_kv_attention_quant_gb300/csrc/rope_consts.h",
                          "quantized_kv_attention_quant_gb300/csrc/kvq_internal.h",
                          "quantized_kv_attention_quant_gb300/csrc/kvq_qprep.cuh",
                          "quantized_kv_attention_quant_gb300/csrc/kvq_append.cuh",
                          "include/kvq.h"],
}


_C_TOKENS = re.compile(r'"(?:\\.|[^"\\\n])*"|\'(?:\\.|[^\'\\\n])*\'|/\*.*?\*/|//[^\n]*', re.S)


def _code_only(text: str) -> str:
    """C/C++/CUDA source with comments removed and whitespace collapsed
    (string and character literals kept as they are)."""
    def keep(m):
        t = m.group(0)
        return t if t[0] in "\"'" else " "
    return " ".join(_C_TOKENS.sub(keep, text).split())


def source_hash(kernel: str) -> str | None:
    """Hash of the code (comments and layout aside) of a kernel's sources."""
    files = KERNEL_SOURCES.get(kernel)
    if not files:
        return None
    h = hashlib.sha256()
    for f in files:
        h.update(f.encode() + b"\0")
        h.update(_code_only(open(os.path.join(ROOT, f), encoding="utf-8").read()).encode() + b"\0")
    return h.hexdigest()[:16]


def traffic_for(kernel: str, key: str, algorithmic_per_launch: float):
    """DRAM bytes per launch of `kernel` from the committed ncu summaries, if
    they were taken on the current kernel sources: the traffic/algorithmic
    ratio measured on one launch (entry `key`, e.g. the cache bit width),
    applied to this launch's algorithmic bytes."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    e = t.get(kernel, {}).get(key)
    if not e or e.get("source_hash") is None or e.get("source_hash") != source_hash(kernel):
        return None
    if e.get("traffic_over_algorithmic") is not None:
        return float(e["traffic_over_algorithmic"]) * algorithmic_per_launch
    return None


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
# distributed plumbing (one process per GPU; replicas of independent work)
# ----------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)


def dist_barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def dist_max(value: float, world: int, device) -> float:
    """Max of a per-rank scalar over all ranks (timing metadata only)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(tokens_per_rank_step: float, ms_local: float, steps: int, world: int, device):
    """(tokens/s of the whole job, ms per step): every rank processes its own
    sequences (weak scaling); the job takes as long as the slowest rank."""
    ms = dist_max(ms_local, world, device)
    ms_step = ms / steps
    return tokens_per_rank_step * world / (ms_step / 1e3), ms_step


# ----------------------------------------------------------------------------
# the GPU arm
# ----------------------------------------------------------------------------

def build_workload(name: str, rank: int, device):
    from quantized_kv_attention_quant_gb300 import harness
    if name in ("stack42", "stack42-e4b"):
        wl = W.workload_stack_decode() if name == "stack42" else W.workload_stack_decode_e4b_bits()
        if rank:
            wl = W.StackWorkload(wl.name, wl.seed + 100 * rank, wl.lengths, wl.donor_bits)
        case = harness.StackCase(wl, device=device, out_f32=False)
        calls = []           # (kind, case) in step order, for e2e and accounting
        for i, d, c in case.layers:
            calls.append((i < W.N_DONORS, c))
        full_bytes = 0
        kv_bytes = 0
        for i, d, c in case.layers:
            spec = c.spec
            by = sum(visible_keys(p, spec.window) * rb_pair(spec.head_dim, b)
                     for p, b in zip(c.wl.filled, c.wl.bits)) * spec.n_kv_heads
            kv_bytes += by
            if spec.window == 0:
                full_bytes += by
        info = {"tokens": wl.n_seqs, "kv_bytes": kv_bytes, "dominant_bytes": full_bytes,
                "dominant": "decode_kernel<512> (full-attention layers)",
                "launches": 42 * 3, "config": {              # 24 donor calls fused with their append
                    "workload": "42-layer mixed decode step, 64 ragged sequences (lengths U[1024,32768]), "
                                "sliding 8q/2kv D256 W512 + full 16q/1kv D512 K=V rope 128, 4/8-bit group 64"
                                + (" (per-donor bits from the seed)" if name == "stack42" else
                                   " (per-donor bits of the e4b layer table: full-layer reads mostly 4-bit)"),
                    "n_seqs": wl.n_seqs, "layers": 42, "kv_donor_layers": 24}}
        return case, calls, info
    if name in ("tiny", "sliding16", "full32k", "full32k-8bit", "full32k-rot"):
        if name == "full32k-8bit":          # the full32k shape with 8-bit caches
            base = W.workload_full_keqv_decode()
            wl = W.DecodeWorkload(base.name + "-8bit", base.seed, base.layer, base.filled, [8] * base.n_seqs)
        elif name == "full32k-rot":         # the full32k shape with the deferred TurboQuant read
            wl = W.workload_full_keqv_rotated_decode()
        else:
            wl = W.WORKLOADS[name]()
        case = harness.DecodeCase(wl, device=device, out_f32=False)
        spec = wl.layer
        by = sum(visible_keys(p, spec.window) * rb_pair(spec.head_dim, b)
                 for p, b in zip(wl.filled, wl.bits)) * spec.n_kv_heads
        info = {"tokens": wl.n_seqs, "kv_bytes": by, "dominant_bytes": by,
                "dominant": f"decode_kernel<{spec.head_dim}>", "launches": 3,    # one fused append + read
                "config": {"workload": wl.name, "n_seqs": wl.n_seqs}}
        return case, [(True, case)], info
    if name == "mixed":
        dwl, pwl = W.workload_mixed_step()
        case = harness.MixedCase([dwl, pwl], device=device, out_f32=False)
        spec = dwl.layer
        dec_by = sum(visible_keys(p, spec.window) * rb_pair(spec.head_dim, b)
                     for p, b in zip(dwl.filled, dwl.bits)) * spec.n_kv_heads
        # the window group reads each sequence's keys once: the window before
        # its first row through its last row
        win_by = sum(min(pwl.filled[s] + pwl.chunk[s], spec.window + pwl.chunk[s] - 1) *
                     rb_pair(spec.head_dim, pwl.bits[s]) for s in range(pwl.n_seqs)) * spec.n_kv_heads
        info = {"tokens": dwl.n_seqs + int(sum(pwl.chunk)), "kv_bytes": dec_by + win_by,
                "dominant_bytes": dec_by + win_by,
                "dominant": "attn_mixed call (decode group: decode_kernel<256>; window group: "
                            "prompt_prep_kernel<256> + prompt_tc_kernel<256>)",
                "launches": 2 + 3 + 2, "mixed": True,
                "config": {"workload": "mixed step of one sliding layer (8q/2kv D256 W512): decode group of "
                                       f"{dwl.n_seqs} sequences (lengths U[1024,8192]) + window group of 2 prompt "
                                       "chunks of 256 rows, one attn_mixed call",
                           "n_seqs": dwl.n_seqs + pwl.n_seqs, "decode_rows": dwl.n_seqs,
                           "window_rows": int(sum(pwl.chunk))}}
        return case, [(True, case)], info
    if name == "mixed-verify":
        dwl, vwl = W.workload_mixed_verify()
        case = harness.MixedCase([dwl, vwl], device=device, out_f32=False)
        spec = dwl.layer
        dec_by = sum(visible_keys(p, spec.window) * rb_pair(spec.head_dim, b)
                     for p, b in zip(dwl.filled, dwl.bits)) * spec.n_kv_heads
        # every verify row reads its own window (the rows of a sequence share
        # most of their keys, read once from HBM and again from L2)
        ver_by = sum(sum(visible_keys(vwl.filled[s] + t, spec.window) for t in range(vwl.chunk[s])) *
                     rb_pair(spec.head_dim, vwl.bits[s]) for s in range(vwl.n_seqs)) * spec.n_kv_heads
        info = {"tokens": dwl.n_seqs + int(sum(vwl.chunk)), "kv_bytes": dec_by + ver_by,
                "dominant_bytes": dec_by + ver_by,
                "dominant": "attn_mixed call: both groups in one grouped launch of qprep_grouped_kernel<256>, "
                            "decode_grouped_kernel<256>, combine_grouped_kernel<256>",
                "launches": 2 + 3, "mixed": True,
                "config": {"workload": "verify step of one sliding layer (8q/2kv D256 W512): decode group of "
                                       f"{dwl.n_seqs} sequences + verify group of {vwl.n_seqs} sequences x "
                                       f"{vwl.chunk[0]} drafted rows (lengths U[1024,8192]), one attn_mixed call",
                           "n_seqs": dwl.n_seqs + vwl.n_seqs, "decode_rows": dwl.n_seqs,
                           "window_rows": int(sum(vwl.chunk))}}
        return case, [(True, case)], info
    if name in ("prefill", "prefill-full"):
        wl = W.workload_prefill_chunk() if name == "prefill" else W.workload_prefill_full()
        case = harness.PrefillCase(wl, device=device, out_f32=False)
        spec = wl.layer
        rows = sum(wl.chunk)
        flops = 0
        for s in range(wl.n_seqs):
            for t in range(wl.chunk[s]):
                flops += 4 * spec.n_q_heads * spec.head_dim * visible_keys(wl.filled[s] + t, spec.window)
        # head_dim 512 takes the row path: the append, then q prep, the
        # decode kernel over every row and the merge
        row_path = spec.head_dim > 256
        info = {"tokens": rows, "flops": flops, "kv_bytes": 0, "dominant_bytes": 0,
                "dominant": (f"decode_kernel<{spec.head_dim}> (row path)" if row_path
                             else f"prompt_tc_kernel<{spec.head_dim}> (tcgen05)"),
                "launches": 4 if row_path else 2,     # sliding: q prep, append, dequantization in one grid; the read
                "config": {"workload": wl.name, "n_seqs": wl.n_seqs, "rows": rows}}
        return case, [(True, case)], info
    if name == "train42":
        sliding, _ = W.workload_train_prefix_shared()
        blocks = sliding.blocks
        case = harness.TrainStackCase(blocks, seed=sliding.seed, device=device, out_f32=False)
        calls = [(i < W.N_DONORS, c) for i, _, c in case.layers]
        flops = sum(4 * c.spec.n_q_heads * c.spec.head_dim * train_visible_total(blocks, c.spec.window)
                    for _, c in calls)
        info = {"tokens": case.n_rows, "flops": flops, "kv_bytes": 0, "dominant_bytes": 0,
                "dominant": "train_tc_kernel<256|512> (tcgen05)",
                "launches": 42 * 2,                   # donors' K/V prep in the q prep's grid
                "config": {"workload": "training forward's stateless read over the 42-layer stack, one packed "
                                       f"sequence of {case.n_rows} rows: a prefix of {blocks[0]} rows shared by "
                                       f"{len(blocks) - 1} branches of {blocks[1]} (block-sparse mask), sliding "
                                       "8q/2kv D256 W512 + full 16q/1kv D512 K=V; plain bf16 keys and values",
                           "rows": case.n_rows, "layers": 42, "kv_donor_layers": 24,
                           "l2": "keys and values of a layer (<= 8 MB) are L2-resident"}}
        return case, calls, info
    raise SystemExit(f"unknown workload {name}")


def train_visible_total(blocks, window: int) -> int:
    """Keys read by all rows of a prefix-shared layout: a prefix row t reads
    the prefix up to itself, a branch row j the prefix and its branch up to
    position P + j (windowed on sliding layers)."""
    P = blocks[0]
    total = 0
    for t in range(P):
        total += t + 1 - (max(0, t - window + 1) if window > 0 else 0)
    for L in blocks[1:]:
        for j in range(L):
            lp = P + j
            lo = max(0, lp - window + 1) if window > 0 else 0
            total += max(0, P - lo) + (lp - max(lo, P) + 1)
    return total


METRIC = {"prefill": "prefill tokens/s", "prefill-full": "prefill tokens/s", "mixed": "mixed-step tokens/s (decode tokens + window rows)",
          "mixed-verify": "mixed-step tokens/s (decode tokens + window rows)",
          "train42": "training-read tokens/s"}


FUSED_CALL = {"DecodeCase": "attn_decode_append", "PrefillCase": "attn_prefill_append",
              "TrainCase": "attn_train_donor_forward"}


def fusable(donor, c) -> bool:
    """A decode donor's append and attention run as one attn_decode_append."""
    return donor and hasattr(c, "append_attend")


def run_call(donor, c, stream=None, fused=True):
    if fused and fusable(donor, c):
        c.append_attend(stream)
        return
    if donor:
        c.append(stream)
    c.attend(stream)


def step_calls(calls, stream=None, fused=True):
    for donor, c in calls:
        run_call(donor, c, stream, fused)


def call_bytes(c) -> int:
    """Algorithmic KV bytes one attention call of a DecodeCase reads."""
    spec = c.spec
    return sum(visible_keys(p, spec.window) * rb_pair(spec.head_dim, b)
               for p, b in zip(c.wl.filled, c.wl.bits)) * spec.n_kv_heads


def measure(workload, case, calls, info, K, warmup, device, world, with_breakdown=True):
    """Warm-up, then K steps captured in one CUDA graph and replayed once
    between CUDA events.  Events captured around each attention call of the
    dominant kernel give its duration.  Returns a dict of timings."""
    import torch
    for _ in range(warmup):
        step_calls(calls)                      # eager (first calls also set kernel attributes)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream(device=device)
    full_calls = ([c for _, c in calls if c.spec.window == 0] if workload.startswith("stack42")
                  else [c for _, c in calls])

    def ev_pair():
        return (torch.cuda.Event(enable_timing=True, external=True),
                torch.cuda.Event(enable_timing=True, external=True))
    try:
        ev = [[ev_pair() for _ in full_calls] for _ in range(K)]
        # every other call too, for the step breakdown (appends outside a fused
        # call, other attention calls)
        ev_app = [[ev_pair() for donor, c in calls if donor and not fusable(donor, c)] for _ in range(K)]
        ev_oth = [[ev_pair() for _, c in calls if c not in full_calls] for _ in range(K)]
        have_inner = True
    except TypeError:
        ev, ev_app, ev_oth, have_inner = None, None, None, False
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        step_calls(calls)                      # one more warm-up on the capture stream
    torch.cuda.synchronize()

    def capture(g, all_events):
        # all_events: time every call (the events break the launch overlap
        # between calls, so that graph is replayed apart from the timed one)
        with torch.cuda.graph(g, stream=stream):
            for k in range(K):
                j = ja = jo = 0
                for donor, c in calls:
                    fused = fusable(donor, c)
                    if donor and not fused:
                        if all_events:
                            ev_app[k][ja][0].record()
                        c.append()
                        if all_events:
                            ev_app[k][ja][1].record()
                            ja += 1
                    inner = have_inner and c in full_calls
                    pair = ev[k][j] if inner else (ev_oth[k][jo] if all_events else None)
                    if pair:
                        pair[0].record()
                    if fused:
                        c.append_attend()
                    else:
                        c.attend()
                    if pair:
                        pair[1].record()
                        if inner:
                            j += 1
                        else:
                            jo += 1
        torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    capture(graph, False)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    replay_stream = torch.cuda.current_stream()     # graph.replay() launches here
    with ClockSampler(device.index) as clk:
        dist_barrier(world, device)
        torch.cuda.synchronize()
        t0.record(replay_stream)
        graph.replay()
        t1.record(replay_stream)
        torch.cuda.synchronize()
        dist_barrier(world, device)
    res = {"ms_total": t0.elapsed_time(t1), "clocks": clk.summary(), "full_calls": full_calls}
    if have_inner:
        res["dom_ms"] = sum(x.elapsed_time(y) for row in ev for x, y in row) / K
        # per dominant call (the same call in every step), for splits by bit width
        res["dom_call_ms"] = [sum(ev[k][j][0].elapsed_time(ev[k][j][1]) for k in range(K)) / K
                              for j in range(len(full_calls))]
    del graph
    if have_inner and not info.get("mixed"):
        # the dominant kernel alone: the same steps, with the library recording
        # an event pair right around each dominant call's attention kernel
        # (kvq_profile_next_read; these records remove that kernel's overlap
        # with its neighbours, so this graph is replayed apart from the timed one)
        from quantized_kv_attention_quant_gb300 import kvq_profile_next_read
        evk = [[ev_pair() for _ in full_calls] for _ in range(K)]
        with torch.cuda.stream(stream):
            for row in evk:
                for x, y in row:                 # create the events before the capture
                    x.record()
                    y.record()
        torch.cuda.synchronize()
        g_k = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_k, stream=stream):
            for k in range(K):
                j = 0
                for donor, c in calls:
                    if c in full_calls:
                        kvq_profile_next_read(*evk[k][j])
                        j += 1
                    run_call(donor, c)
        torch.cuda.synchronize()
        g_k.replay()
        torch.cuda.synchronize()
        res["kern_call_ms"] = [sum(evk[k][j][0].elapsed_time(evk[k][j][1]) for k in range(K)) / K
                               for j in range(len(full_calls))]
        res["kern_ms"] = sum(res["kern_call_ms"])
        del g_k
    if any(fusable(d, c) for d, c in calls) and not info.get("mixed"):
        # the same steps with every donor's append as its own kv_quant_append
        # call before its attn_decode (the same timing events around the
        # dominant calls as the timed graph)
        g_sep = torch.cuda.CUDAGraph()
        ev_sep = [[ev_pair() for _ in full_calls] for _ in range(K)] if have_inner else None
        with torch.cuda.graph(g_sep, stream=stream):
            for k in range(K):
                j = 0
                for donor, c in calls:
                    if donor:
                        c.append()
                    pair = ev_sep[k][j] if (ev_sep and c in full_calls) else None
                    if pair:
                        pair[0].record()
                    c.attend()
                    if pair:
                        pair[1].record()
                        j += 1
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(replay_stream)
        g_sep.replay()
        a1.record(replay_stream)
        torch.cuda.synchronize()
        res["separate_append_ms"] = a0.elapsed_time(a1) / K
        del g_sep
    if info.get("mixed"):
        # the same steps with every group as its own call on one stream
        # (with the same timing events around the attention calls as the
        # timed graph, so that both graphs have the same structure)
        g_ser = torch.cuda.CUDAGraph()
        ev_ser = [ev_pair() for _ in range(K)] if have_inner else None
        with torch.cuda.graph(g_ser, stream=stream):
            for k in range(K):
                for _, c in calls:
                    c.append()
                    if ev_ser:
                        ev_ser[k][0].record()
                    c.attend_serial()
                    if ev_ser:
                        ev_ser[k][1].record()
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(replay_stream)
        g_ser.replay()
        a1.record(replay_stream)
        torch.cuda.synchronize()
        res["serial_ms"] = a0.elapsed_time(a1) / K
        del g_ser
    if have_inner and with_breakdown:
        # per-call breakdown from a separate replay with events around every call
        graph_bd = torch.cuda.CUDAGraph()
        capture(graph_bd, True)
        graph_bd.replay()
        torch.cuda.synchronize()
        res["breakdown"] = {"dominant_calls_ms": sum(x.elapsed_time(y) for row in ev for x, y in row) / K,
                            "other_attention_calls_ms": sum(x.elapsed_time(y) for row in ev_oth for x, y in row) / K,
                            "append_calls_ms": sum(x.elapsed_time(y) for row in ev_app for x, y in row) / K}
        del graph_bd
    res["status_ok"] = all(all(w == 0 for w in (c.status_words() if hasattr(c, "status_words")
                                                 else [c.status_word()])) for _, c in calls)
    return res


def roofline(workload, info, res, peaks):
    """The dominant kernel's roofline object: algorithmic work over the
    kernel's own launch durations (event pairs the library records right
    around it, `kern_ms`), and beside it the same over the whole calls (q
    prep, the donor's append, the kernel and the merge: events around each
    call inside the timed graph, `dom_ms`)."""
    dom_ms = res.get("dom_ms")
    if not dom_ms:
        return None
    kern_ms = res.get("kern_ms") or dom_ms
    n_calls = max(1, len(res["full_calls"]))
    if workload in ("prefill", "prefill-full", "train42"):
        achieved = info["flops"] / (kern_ms / 1e3) / 1e12
        call = info["flops"] / (dom_ms / 1e3) / 1e12
        return {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"], "traffic": None,
                "peak_source": peaks["source"] + " bf16 burst (f16 runs at the bf16 rate)",
                "kernel": info["dominant"], "launch_ms": kern_ms / n_calls,
                "call": {"achieved": call, "frac": call / peaks["bf16_tflops"], "ms": dom_ms / n_calls}}
    achieved = info["dominant_bytes"] / (kern_ms / 1e3) / 1e9
    call = info["dominant_bytes"] / (dom_ms / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "frac_of_nominal_8000": achieved / 8000.0,
            "traffic": None, "peak_source": peaks["source"], "kernel": info["dominant"],
            "launch_ms": kern_ms / n_calls,
            "call": {"achieved": call, "frac": call / peaks["hbm_gbs"], "ms": dom_ms / n_calls}}
    # DRAM traffic per launch from the committed ncu summaries, keyed by the
    # kernel's sources and the cache bit width (weighted by each call's bytes)
    calls = res["full_calls"]
    if "512" in info["dominant"] and all(hasattr(c, "wl") for c in calls):
        tr = 0.0
        for c in calls:
            t = traffic_for("decode_kernel_512", f"{c.wl.bits[0]}bit", call_bytes(c))
            if t is None:
                tr = None
                break
            tr += t
        roof["traffic"] = None if tr is None else tr / n_calls
    return roof


def bit_split(res, peaks):
    """The dominant kernel's bytes, time and HBM fraction per cache bit width
    (kernel alone; `call_*`: the whole calls)."""
    out = {}
    kern = res.get("kern_call_ms") or res.get("dom_call_ms", [])
    for c, ms, cms in zip(res["full_calls"], kern, res.get("dom_call_ms", [])):
        b = c.wl.bits[0]
        o = out.setdefault(f"{b}bit", {"calls": 0, "bytes": 0, "ms": 0.0, "call_ms": 0.0})
        o["calls"] += 1
        o["bytes"] += call_bytes(c)
        o["ms"] += ms
        o["call_ms"] += cms
    for o in out.values():
        o["achieved_gbs"] = o["bytes"] / (o["ms"] / 1e3) / 1e9
        o["frac"] = o["achieved_gbs"] / peaks["hbm_gbs"]
        o["ms_per_call"] = o["ms"] / o["calls"]
        o["call_frac"] = o["bytes"] / (o["call_ms"] / 1e3) / 1e9 / peaks["hbm_gbs"]
    return out


def sub_result(name, K, warmup, device, peaks):
    """One more workload timed in the same run (CUDA events on a graph of K
    steps): its own rate and its dominant kernel's roofline."""
    import torch
    case, calls, info = build_workload(name, 0, device)
    torch.cuda.synchronize()
    res = measure(name, case, calls, info, K, warmup, device, 1, with_breakdown=False)
    ms_step = res["ms_total"] / K
    out = {"metric": METRIC.get(name, "decode-attention tokens/s"), "value": info["tokens"] / (ms_step / 1e3),
           "unit": "tokens/s", "ms_per_step": ms_step, "workload": info["config"]["workload"],
           "roofline": roofline(name, info, res, peaks), "device_status_clean": res["status_ok"],
           "clocks": res["clocks"]}
    if res.get("separate_append_ms") is not None:
        out["separate_append_ms_per_step"] = res["separate_append_ms"]
    if info["kv_bytes"]:
        out["kv_bytes_per_step"] = info["kv_bytes"]
    if name.startswith("stack42") and res.get("dom_call_ms"):
        out["dominant_by_bits"] = bit_split(res, peaks)
    del case, calls
    torch.cuda.empty_cache()
    return out


def run_gpu(args):
    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist_init(world, "nccl")
    case, calls, info = build_workload(args.workload, rank, device)
    torch.cuda.synchronize()
    K = args.steps
    res = measure(args.workload, case, calls, info, K, args.warmup, device, world)
    value, ms_step = whole_job_rate(info["tokens"], res["ms_total"], K, world, device)

    # e2e through the binding with host buffers
    e2e = run_e2e(calls, K, device, info, world)

    peaks = load_peaks()
    roof = roofline(args.workload, info, res, peaks)
    step_gbs = info["kv_bytes"] / (ms_step / 1e3) / 1e9 if info["kv_bytes"] else None

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = run_cpu_baseline(args.workload, steps=1, warmup=0)

    cfg = dict(info["config"])
    cfg.update({"l2": "inputs larger than L2" if info["kv_bytes"] > 129e6 else
                "inputs smaller than L2 (launch-bound case)",
                "kv_bytes_per_step": info["kv_bytes"], "step_kv_gbs": step_gbs,
                "graph": f"{K} steps captured in one CUDA graph", "device_status_clean": res["status_ok"],
                "compute": "packed 4/8-bit codes; f16 tensor-core operands (codes exact), fp32 accumulation"})
    if res.get("serial_ms") is not None:
        cfg["separate_calls_ms_per_step"] = res["serial_ms"]
    fused_calls = sorted({FUSED_CALL[type(c).__name__] for d, c in calls if fusable(d, c)})
    if fused_calls:
        cfg["donor_calls"] = (", ".join(fused_calls) + " (each donor's K/V append and its attention read in one "
                              "call; the append runs beside the q prep in the call's first kernel)")
    if res.get("separate_append_ms") is not None:
        cfg["separate_append_ms_per_step"] = res["separate_append_ms"]
    if res.get("breakdown"):
        cfg["step_breakdown_ms"] = {k: round(v, 4) for k, v in res["breakdown"].items()}
        cfg["step_breakdown_note"] = ("separate replay with events around every call (they slow it down); "
                                      "fused donor appends count with the attention calls")
    if args.workload.startswith("stack42") and res.get("dom_call_ms"):
        cfg["dominant_by_bits"] = bit_split(res, peaks)
    del case, calls
    if args.workload == "stack42" and world == 1 and not args.no_sub_results:
        # the long-context and tensor-core workloads, timed in the same run
        torch.cuda.empty_cache()
        cfg["sub_results"] = {name: sub_result(name, K, args.warmup, device, peaks)
                              for name in ("stack42-e4b", "full32k", "full32k-rot", "prefill", "train42")}
    line = {"metric": METRIC.get(args.workload, "decode-attention tokens/s"),
            "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16 inputs, norm weights 1+N(0,0.1))",
            "config": cfg, "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": info["launches"] * K, "clocks": res["clocks"]}
    if rank == 0:
        print(json.dumps(line), flush=True)


def call_inputs(donor, c):
    """Device inputs a call reads each step (q; plus k/v rows when it appends)."""
    if hasattr(c, "inputs"):
        return c.inputs()
    return [c.q] + ([c.k] + ([c.v] if c.v is not None else []) if donor else [])


def call_outputs(c):
    return c.outputs() if hasattr(c, "outputs") else [c.out]


def run_e2e(calls, K, device, info, world):
    """K steps through the binding; every step copies its q/k/v inputs from
    pinned host memory and its outputs back.  The copies run on two side
    streams, layer by layer, so that they overlap the other layers' calls:
    layer L's inputs land while earlier layers compute, and its output is
    read back while later layers compute.  Events order every buffer reuse
    (a layer's inputs are overwritten only after its call of the previous
    step, its output only after the previous read-back).  The K steps, copies
    included, are captured in one CUDA graph (as the device-side number is)
    and replayed once inside the timed region."""
    import torch
    host_in, host_out = [], []
    for donor, c in calls:
        host_in.append([torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t) for t in call_inputs(donor, c)])
        host_out.append([torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in call_outputs(c)])
    bi = sum(t.numel() * t.element_size() for hs in host_in for t in hs)
    bo = sum(t.numel() * t.element_size() for hs in host_out for t in hs)
    cap = torch.cuda.Stream(device)
    cin, cout = torch.cuda.Stream(device), torch.cuda.Stream(device)
    n = len(calls)

    def steps(k_steps):
        s = torch.cuda.current_stream()
        fork = torch.cuda.Event()
        fork.record(s)
        cin.wait_event(fork)
        cout.wait_event(fork)
        done = [None] * n        # layer L's call of the previous step finished (its inputs are free)
        read = [None] * n        # layer L's output of the previous step copied back
        for _ in range(k_steps):
            ready = []
            with torch.cuda.stream(cin):
                for L, ((donor, c), hs) in enumerate(zip(calls, host_in)):
                    if done[L] is not None:
                        cin.wait_event(done[L])
                    for d, h in zip(call_inputs(donor, c), hs):
                        d.copy_(h, non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(cin)
                    ready.append(ev)
            for L, (donor, c) in enumerate(calls):
                s.wait_event(ready[L])
                if read[L] is not None:
                    s.wait_event(read[L])
                run_call(donor, c)
                ev = torch.cuda.Event()
                ev.record(s)
                done[L] = ev
                cout.wait_event(ev)
                with torch.cuda.stream(cout):
                    for h, d in zip(host_out[L], call_outputs(c)):
                        h.copy_(d, non_blocking=True)
                    ev2 = torch.cuda.Event()
                    ev2.record(cout)
                read[L] = ev2
        for ev in read + done:
            s.wait_event(ev)
        last_in = torch.cuda.Event()
        last_in.record(cin)
        s.wait_event(last_in)

    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        steps(1)                                   # eager warm-up of the same sequence
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        steps(K)
    torch.cuda.synchronize()
    rs = torch.cuda.current_stream()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    dist_barrier(world, device)
    t0.record(rs)
    graph.replay()
    t1.record(rs)
    torch.cuda.synchronize()
    dist_barrier(world, device)
    ms = dist_max(t0.elapsed_time(t1), world, device) / K
    del graph
    return {"value": info["tokens"] * world / (ms / 1e3), "unit": "tokens/s",
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "ms_per_step": ms,
            "copies": "per layer on two side streams overlapping the other layers' calls; K steps in one CUDA graph"}


# ----------------------------------------------------------------------------
# the CPU oracle (reference arm and cpu_baseline)
# ----------------------------------------------------------------------------

def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_cpu_baseline(workload: str, steps: int, warmup: int):
    """The oracle as it stands on the host cores: one single-threaded worker
    process per core, one sampled sequence per worker (sequences spread over
    the workload's length distribution)."""
    cores = host_cores()
    n_all = {"stack42": 64, "stack42-e4b": 64, "tiny": 1, "sliding16": 16, "full32k": 8, "full32k-8bit": 8,
             "full32k-rot": 8}.get(workload, 1)
    nseq = max(1, min(cores, n_all))
    procs = nseq if workload in ("stack42", "stack42-e4b", "tiny", "sliding16", "full32k", "full32k-8bit",
                                 "full32k-rot") else 1
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    cmd = [sys.executable, os.path.join(ROOT, "oracle", "timing.py"), workload, str(steps), str(warmup),
           str(nseq), str(procs)]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, cwd=ROOT, timeout=1800)
    if r.returncode != 0:
        return {"error": r.stderr[-500:]}
    res = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": res["tokens_per_s"], "unit": "tokens/s", "cores": res.get("procs", 1), "kind": "oracle",
            "sample": res["sample"], "ms_per_step": res["ms_per_step"], "host_cores": cores,
            "cpu_model": res.get("cpu_model")}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    res = run_cpu_baseline(args.workload, steps=args.steps, warmup=args.warmup)
    line = {"impl": "reference", "metric": METRIC.get(args.workload, "decode-attention tokens/s"),
            "value": res.get("value"), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": res.get("ms_per_step"),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, same generators as the GPU arm)",
            "config": {"workload": args.workload, "sample": res.get("sample")},
            "cpu_baseline": res,
            "e2e": {"value": res.get("value"), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="stack42",
                    choices=["stack42", "stack42-e4b", "tiny", "sliding16", "full32k", "full32k-8bit",
                             "full32k-rot", "prefill", "prefill-full", "mixed", "mixed-verify", "train42"])
    ap.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sub-results", action="store_true",
                    help="stack42 only: skip timing full32k and prefill in the same run")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
