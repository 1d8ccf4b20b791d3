"""Runs the library on the seeded workloads of `workloads`: allocates the
caches in device memory, fills every cached position through kv_quant_append,
uploads each step's inputs and runs steps.  The tests and bench.py drive the
GPU path through these classes; the arithmetic happens only in libkvq.so.
"""
from __future__ import annotations

import concurrent.futures as cf
import multiprocessing as mp
import os

import numpy as np
import torch

import workloads as W

from . import (KVQ_PHASE_DECODE, KVQ_PHASE_WINDOW, attn_decode, attn_decode_append, attn_decode_workspace_bytes,
               attn_group, attn_mixed, attn_prefill_append, attn_prefill_chunk, attn_prefill_workspace_bytes,
               attn_train_donor_forward, attn_train_forward, attn_train_workspace_bytes, kv_quant_append,
               kvq_train_kv_prep, layer as make_layer)
from .cache import LayerCaches


def kvq_layer(spec: W.LayerSpec, rot_signs=None):
    """The library's layer descriptor; rot_signs: the device int8 signs of a
    rotated layer (spec.kv_rotation), else None."""
    return make_layer(spec.n_q_heads, spec.n_kv_heads, spec.head_dim, spec.window, spec.rope_dims,
                      spec.rope_theta, spec.rms_eps, spec.k_eq_v, rot_signs=rot_signs)


def dev_signs(inp, device):
    """The layer's rotation signs on the device (int8), or None."""
    return None if inp.get("rot") is None else torch.from_numpy(np.ascontiguousarray(inp["rot"])).to(device)


def dev_bits(a: np.ndarray, device) -> torch.Tensor:
    """Upload bf16 bit patterns (uint16) as an int16 device tensor."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device)


def dev_i32(values, device) -> torch.Tensor:
    return torch.tensor(np.asarray(values, dtype=np.int32), device=device)


_POOL = None


def _gen_pool():
    """Worker processes for drawing cache rows (spawned, so safe to start after
    CUDA is initialised in this process)."""
    global _POOL
    if _POOL is None:
        n = max(1, min(16, (os.cpu_count() or 2) - 1))
        _POOL = cf.ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn"))
    return _POOL


def fill_caches(caches: LayerCaches, spec: W.LayerSpec, seed: int, layer_id: int, positions_of,
                k_w: torch.Tensor, device, max_rows_per_call: int = 1 << 20, keep_prepped=False, lay=None):
    """Append the raw rows of every cached position of every sequence.

    positions_of(s) -> int array of the positions resident before the step.
    Returns {s: prepped [2, n, Hkv, D] uint16} when keep_prepped, else {}."""
    lay = lay if lay is not None else kvq_layer(spec)
    desc_size = 56
    kept = {}
    s = 0
    n = caches.n_seqs
    while s < n:
        # group sequences into one call up to max_rows_per_call rows
        group, rows = [], 0
        while s < n:
            pos = positions_of(s)
            if group and rows + len(pos) > max_rows_per_call:
                break
            group.append((s, pos))
            rows += len(pos)
            s += 1
        if rows == 0:
            continue
        ks, vs, offs, starts = [], [], [0], []
        jobs = [(seed, layer_id, si, spec, pos) for si, pos in group]
        if rows >= 65536 and len(group) > 1:
            results = list(_gen_pool().map(W.cache_rows_job, jobs))
        else:
            results = [W.cache_rows_job(j) for j in jobs]
        for (si, pos), (k, v) in zip(group, results):
            ks.append(k)
            if v is not None:
                vs.append(v)
            offs.append(offs[-1] + len(pos))
            starts.append(int(pos[0]) if len(pos) else 0)
        k_raw = dev_bits(np.concatenate(ks), device)
        v_raw = dev_bits(np.concatenate(vs), device) if vs else None
        prepped = None
        if keep_prepped:
            prepped = torch.empty((2, rows, spec.n_kv_heads, spec.head_dim), dtype=torch.int16, device=device)
        first = group[0][0]
        # the descriptor array of this group starts at sequence `first`
        kv_quant_append(lay, caches.desc.data_ptr() + first * desc_size, len(group), dev_i32(offs, device),
                        dev_i32(starts, device), rows, k_raw, v_raw, k_w, prepped)
        if keep_prepped:
            host = prepped.cpu().numpy().view(np.uint16)
            for j, (si, _) in enumerate(group):
                kept[si] = host[:, offs[j]:offs[j + 1]]
        del k_raw, v_raw
    return kept


class DecodeCase:
    """One decode step of one layer (DecodeWorkload): every sequence appends its
    new token's K/V row, then attends with one query token."""

    def __init__(self, wl: W.DecodeWorkload, device="cuda", keep_prepped=False, out_f32=True,
                 caches: LayerCaches | None = None, fill=True, keep_fill=None):
        self.wl, self.spec, self.device = wl, wl.layer, device
        spec, n = wl.layer, wl.n_seqs
        inp = W.layer_inputs(wl.seed, wl.layer_id, spec, n, n)
        self.rot = dev_signs(inp, device)
        self.lay = kvq_layer(spec, self.rot)
        self.host_inputs = inp
        self.q_w = dev_bits(inp["q_w"], device)
        self.k_w = dev_bits(inp["k_w"], device)
        self.q = dev_bits(inp["q"], device)
        self.k = dev_bits(inp["k"], device)
        self.v = dev_bits(inp["v"], device) if inp["v"] is not None else None
        self.caches = caches or LayerCaches(spec.n_kv_heads, spec.head_dim, wl.bits,
                                            [wl.capacity(s) for s in range(n)], device)
        self.fill_prepped = {}
        if fill:
            self.fill_prepped = fill_caches(self.caches, spec, wl.seed, wl.layer_id, wl.cached_positions,
                                            self.k_w, device,
                                            keep_prepped=keep_prepped if keep_fill is None else keep_fill,
                                            lay=self.lay)
        self.pos = dev_i32(wl.filled, device)
        self.offs = dev_i32(np.arange(n + 1), device)
        self.max_pos = int(max(wl.filled))
        self.ws_bytes = attn_decode_workspace_bytes(self.lay, n, self.max_pos)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)
        self.out_f32 = out_f32
        self.out = torch.empty((n, spec.n_q_heads, spec.head_dim),
                               dtype=torch.float32 if out_f32 else torch.int16, device=device)
        self.keep_prepped = keep_prepped
        self.q_prepped = torch.empty_like(self.q) if keep_prepped else None
        self.kv_prepped = (torch.empty((2, n, spec.n_kv_heads, spec.head_dim), dtype=torch.int16, device=device)
                           if keep_prepped else None)

    def append(self, stream=None):
        kv_quant_append(self.lay, self.caches.desc, self.wl.n_seqs, self.offs, self.pos, self.wl.n_seqs,
                        self.k, self.v, self.k_w, self.kv_prepped, stream)

    def attend(self, stream=None, caches: LayerCaches | None = None):
        c = caches or self.caches
        attn_decode(self.lay, c.desc, self.wl.n_seqs, self.pos, self.max_pos, self.q, self.q_w, self.out,
                    self.out_f32, self.q_prepped, self.ws, self.ws_bytes, stream)

    def append_attend(self, stream=None):
        """append + attend as one attn_decode_append call."""
        attn_decode_append(self.lay, self.caches.desc, self.wl.n_seqs, self.pos, self.max_pos, self.q, self.k,
                           self.v, self.q_w, self.k_w, self.out, self.out_f32, self.q_prepped, self.kv_prepped,
                           self.ws, self.ws_bytes, stream)

    def step(self, stream=None):
        self.append(stream)
        self.attend(stream)

    def status_word(self) -> int:
        return int(self.ws[:4].cpu().numpy().view(np.uint32)[0])


class PrefillCase:
    """One prompt chunk of one layer (PrefillWorkload): every sequence appends
    its chunk's K/V rows, then all chunk rows attend."""

    def __init__(self, wl: W.PrefillWorkload, device="cuda", keep_prepped=False, out_f32=True, fill=True):
        self.wl, self.spec, self.device = wl, wl.layer, device
        spec, n = wl.layer, wl.n_seqs
        self.rot = dev_signs(W.layer_inputs(wl.seed, wl.layer_id, spec, 0, 0), device)
        self.lay = kvq_layer(spec, self.rot)
        rows = int(sum(wl.chunk))
        self.n_rows = rows
        self.host_inputs = []
        qs, ks, vs = [], [], []
        for s in range(n):
            inp = W.layer_inputs(wl.seed, wl.layer_id, spec, wl.chunk[s], wl.chunk[s], seq=s)
            self.host_inputs.append(inp)
            qs.append(inp["q"]); ks.append(inp["k"])
            if inp["v"] is not None:
                vs.append(inp["v"])
        w = self.host_inputs[0] if n else W.layer_inputs(wl.seed, wl.layer_id, spec, 0, 0)
        self.q_w = dev_bits(w["q_w"], device)
        self.k_w = dev_bits(w["k_w"], device)
        self.q = dev_bits(np.concatenate(qs), device)
        self.k = dev_bits(np.concatenate(ks), device)
        self.v = dev_bits(np.concatenate(vs), device) if vs else None
        self.caches = LayerCaches(spec.n_kv_heads, spec.head_dim, wl.bits,
                                  [wl.capacity(s) for s in range(n)], device)
        self.fill_prepped = {}
        if fill:
            self.fill_prepped = fill_caches(self.caches, spec, wl.seed, wl.layer_id, wl.cached_positions,
                                            self.k_w, device, keep_prepped=keep_prepped, lay=self.lay)
        self.offs = dev_i32(np.concatenate([[0], np.cumsum(wl.chunk)]), device)
        self.start = dev_i32(wl.filled, device)
        self.max_rows = int(max(wl.chunk))
        self.ws_bytes = attn_prefill_workspace_bytes(self.lay, n, rows, self.max_rows)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)
        self.out_f32 = out_f32
        self.out = torch.empty((rows, spec.n_q_heads, spec.head_dim),
                               dtype=torch.float32 if out_f32 else torch.int16, device=device)
        self.q_prepped = torch.empty_like(self.q) if keep_prepped else None
        self.kv_prepped = (torch.empty((2, rows, spec.n_kv_heads, spec.head_dim), dtype=torch.int16, device=device)
                           if keep_prepped else None)

    def append(self, stream=None):
        kv_quant_append(self.lay, self.caches.desc, self.wl.n_seqs, self.offs, self.start, self.n_rows,
                        self.k, self.v, self.k_w, self.kv_prepped, stream)

    def attend(self, stream=None):
        attn_prefill_chunk(self.lay, self.caches.desc, self.wl.n_seqs, self.offs, self.start, self.n_rows,
                           self.max_rows, self.q, self.q_w, self.out, self.out_f32, self.q_prepped, self.ws,
                           self.ws_bytes, stream)

    def append_attend(self, stream=None):
        """append + attend as one attn_prefill_append call."""
        attn_prefill_append(self.lay, self.caches.desc, self.wl.n_seqs, self.offs, self.start, self.n_rows,
                            self.max_rows, self.q, self.k, self.v, self.q_w, self.k_w, self.out, self.out_f32,
                            self.q_prepped, self.kv_prepped, self.ws, self.ws_bytes, stream)

    def step(self, stream=None):
        self.append(stream)
        self.attend(stream)

    def status_word(self) -> int:
        return int(self.ws[:4].cpu().numpy().view(np.uint32)[0])


class MixedCase:
    """Groups of one layer in one attn_mixed call: DecodeWorkload groups (one
    query row per sequence) and PrefillWorkload groups (prompt chunks or
    verify windows), each group with its own caches, bit widths and positions.  The groups
    must share the layer spec, seed and layer id (hence the q norm weight)."""

    def __init__(self, workloads, device="cuda", keep_prepped=False, out_f32=True):
        self.cases = []
        for wl in workloads:
            if isinstance(wl, W.DecodeWorkload):
                self.cases.append(DecodeCase(wl, device, keep_prepped=keep_prepped, out_f32=out_f32))
            else:
                self.cases.append(PrefillCase(wl, device, keep_prepped=keep_prepped, out_f32=out_f32))
        first = self.cases[0]
        self.spec, self.lay, self.q_w, self.out_f32 = first.spec, first.lay, first.q_w, out_f32
        for c in self.cases[1:]:
            assert c.wl.seed == first.wl.seed and c.wl.layer_id == first.wl.layer_id and c.spec == first.spec

    def groups(self):
        gs = []
        for c in self.cases:
            if isinstance(c, DecodeCase):
                gs.append(attn_group(KVQ_PHASE_DECODE, c.caches.desc, c.wl.n_seqs, None, c.pos, 0, c.max_pos, 0,
                                     c.q, c.out, c.q_prepped, c.ws, c.ws_bytes))
            else:
                gs.append(attn_group(KVQ_PHASE_WINDOW, c.caches.desc, c.wl.n_seqs, c.offs, c.start, c.n_rows, 0,
                                     c.max_rows, c.q, c.out, c.q_prepped, c.ws, c.ws_bytes))
        return gs

    def append(self, stream=None):
        for c in self.cases:
            c.append(stream)

    def attend(self, stream=None):
        attn_mixed(self.lay, self.groups(), self.q_w, self.out_f32, stream)

    def attend_serial(self, stream=None):
        for c in self.cases:
            c.attend(stream)

    def step(self, stream=None):
        self.append(stream)
        self.attend(stream)

    def inputs(self):
        return [t for c in self.cases for t in (c.q, c.k) + ((c.v,) if c.v is not None else ())]

    def outputs(self):
        return [c.out for c in self.cases]

    def status_words(self):
        return [c.status_word() for c in self.cases]


class StackCase:
    """Decode step over the 42-layer stack (StackWorkload): donors 0..23 append
    and attend their own caches; layers 24..41 attend their donor's cache.

    Layers listed in `inspect` also write their prepped q rows and their new
    K/V rows (not the cached rows of the fill) for comparison."""

    def __init__(self, wl: W.StackWorkload, device="cuda", out_f32=True, inspect=()):
        self.wl = wl
        self.layers = []
        self.donor_case = {}
        for i in range(W.N_LAYERS):
            d = W.stack_cache_layer(i)
            view = wl.decode_view(i)
            keep = i in inspect
            if i < W.N_DONORS:
                case = DecodeCase(view, device, out_f32=out_f32, keep_prepped=keep, keep_fill=False)
                self.donor_case[i] = case
            else:
                # a sharer: its own q inputs, the donor's caches, no append
                sv = W.DecodeWorkload(view.name, wl.seed, view.layer, view.filled, view.bits, layer_id=i)
                case = DecodeCase(sv, device, out_f32=out_f32, caches=self.donor_case[d].caches, fill=False,
                                  keep_prepped=keep)
            self.layers.append((i, d, case))

    def step(self, stream=None, fused=True):
        """One step: each donor's append and read as one attn_decode_append
        (fused) or as kv_quant_append + attn_decode; sharers read only."""
        for i, d, case in self.layers:
            if i < W.N_DONORS and fused:
                case.append_attend(stream)
                continue
            if i < W.N_DONORS:
                case.append(stream)
            case.attend(stream)


class TrainCase:
    """The training forward's read of one layer over one packed sequence
    (TrainWorkload): a donor layer preps its plain keys and values, then every
    row attends under the prefix-shared layout.  With `kv` = (k_hat, v_hat) of
    a donor the layer is a KV-sharing one: it reads those and preps none."""

    def __init__(self, wl: W.TrainWorkload, device="cuda", out_f32=True, keep_prepped=False, kv=None,
                 layer_id=0):
        self.wl, self.spec, self.device = wl, wl.layer, device
        spec, T = wl.layer, wl.n_rows
        self.lay = kvq_layer(spec)
        inp = W.layer_inputs(wl.seed, layer_id, spec, T, T)
        self.host_inputs = inp
        self.q_w = dev_bits(inp["q_w"], device)
        self.k_w = dev_bits(inp["k_w"], device)
        self.q = dev_bits(inp["q"], device)
        self.donor = kv is None
        if self.donor:
            self.k = dev_bits(inp["k"], device)
            self.v = dev_bits(inp["v"], device) if inp["v"] is not None else None
            shape = (T, spec.n_kv_heads, spec.head_dim)
            self.k_hat = torch.empty(shape, dtype=torch.int16, device=device)
            self.v_hat = torch.empty(shape, dtype=torch.int16, device=device)
        else:
            self.k_hat, self.v_hat = kv
        self.n_rows = T
        self.n_blocks = len(wl.blocks)
        self.offs = dev_i32(wl.offsets(), device)
        self.max_rows = max(1, min(T, int(max(wl.blocks))))
        self.ws_bytes = attn_train_workspace_bytes(self.lay, T)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)
        self.out_f32 = out_f32
        self.out = torch.empty((T, spec.n_q_heads, spec.head_dim), dtype=torch.float32 if out_f32 else torch.int16,
                               device=device)
        self.q_prepped = torch.empty_like(self.q) if keep_prepped else None

    @property
    def kv(self):
        return self.k_hat, self.v_hat

    def prep_kv(self, stream=None):
        kvq_train_kv_prep(self.lay, self.n_blocks, self.offs, self.n_rows, self.k, self.v, self.k_w, self.k_hat,
                          self.v_hat, stream)

    def attend(self, stream=None):
        attn_train_forward(self.lay, self.n_blocks, self.offs, self.n_rows, self.max_rows, self.q, self.q_w,
                           self.k_hat, self.v_hat, self.out, self.out_f32, self.q_prepped, self.ws, self.ws_bytes,
                           stream)

    def append(self, stream=None):
        """The donor's part of a step (the name the step drivers use)."""
        self.prep_kv(stream)

    def append_attend(self, stream=None):
        """A donor's K/V prep and read as one attn_train_donor_forward call."""
        attn_train_donor_forward(self.lay, self.n_blocks, self.offs, self.n_rows, self.max_rows, self.q, self.k,
                                 self.v, self.q_w, self.k_w, self.k_hat, self.v_hat, self.out, self.out_f32,
                                 self.q_prepped, self.ws, self.ws_bytes, stream)

    def step(self, stream=None, fused=False):
        if self.donor and fused:
            self.append_attend(stream)
            return
        if self.donor:
            self.prep_kv(stream)
        self.attend(stream)

    def status_word(self) -> int:
        return int(self.ws[:4].cpu().numpy().view(np.uint32)[0])


class TrainStackCase:
    """The training forward's reads over the 42-layer stack for one packed
    sequence: donors 0..23 prep their keys and values and attend, layers
    24..41 attend the keys and values of the last donor of their type (as the
    donors hand theirs to their sharers)."""

    def __init__(self, blocks, seed=1007, device="cuda", out_f32=True, keep_prepped=(), name="train-stack"):
        self.layers = []
        donors = {}
        for i in range(W.N_LAYERS):
            spec = W.FULL_KEQV if W.stack_layer_kind(i) == "full" else W.SLIDING
            wl = W.TrainWorkload(f"{name}-layer{i}", seed, spec, list(blocks))
            d = W.stack_cache_layer(i)
            kv = None if i < W.N_DONORS else donors[d].kv
            case = TrainCase(wl, device, out_f32=out_f32, keep_prepped=i in keep_prepped, kv=kv, layer_id=i)
            if i < W.N_DONORS:
                donors[i] = case
            self.layers.append((i, d, case))
        self.n_rows = int(sum(blocks))

    def step(self, stream=None, fused=True):
        for _, _, case in self.layers:
            case.step(stream, fused=fused)
