"""Device memory for quantized KV caches, allocated through torch.

One LayerCaches holds the caches of every sequence of one layer in the layout
include/kvq.h documents, plus the device array of kvq_seq_cache descriptors
the kernels read.  torch is used only as the allocator.
"""
from __future__ import annotations

import numpy as np
import torch

from . import KvqSeqCache

GROUP = 64


class LayerCaches:
    def __init__(self, n_kv_heads: int, head_dim: int, bits, capacity, device="cuda"):
        n = len(bits)
        assert len(capacity) == n
        self.n_kv_heads, self.head_dim = n_kv_heads, head_dim
        self.bits = [int(b) for b in bits]
        self.capacity = [int(c) for c in capacity]
        self.seqs = []
        descs = (KvqSeqCache * max(n, 1))()
        ng = head_dim // GROUP
        for s in range(n):
            b, cap = self.bits[s], self.capacity[s]
            words = head_dim * b // 32
            t = {
                "k_codes": torch.zeros((n_kv_heads, cap, words), dtype=torch.int32, device=device),
                "v_codes": torch.zeros((n_kv_heads, cap, words), dtype=torch.int32, device=device),
                "k_scales": torch.zeros((n_kv_heads, cap, ng), dtype=torch.int16, device=device),
                "k_biases": torch.zeros((n_kv_heads, cap, ng), dtype=torch.int16, device=device),
                "v_scales": torch.zeros((n_kv_heads, cap, ng), dtype=torch.int16, device=device),
                "v_biases": torch.zeros((n_kv_heads, cap, ng), dtype=torch.int16, device=device),
            }
            self.seqs.append(t)
            descs[s] = KvqSeqCache(t["k_codes"].data_ptr(), t["v_codes"].data_ptr(),
                                   t["k_scales"].data_ptr(), t["k_biases"].data_ptr(),
                                   t["v_scales"].data_ptr(), t["v_biases"].data_ptr(), b, cap)
        raw = np.frombuffer(bytes(descs), dtype=np.uint8).copy()
        self.desc = torch.from_numpy(raw).to(device)
        self.n_seqs = n

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for d in self.seqs for t in d.values())

    def host_rows(self, s: int, slots):
        """Packed words (uint32) and scale/bias bit patterns (uint16) of the
        given slots of sequence s: dict name -> array [H, len(slots), ...]."""
        idx = torch.as_tensor(np.asarray(slots, dtype=np.int64), device=self.seqs[s]["k_codes"].device)
        out = {}
        for name, t in self.seqs[s].items():
            a = t.index_select(1, idx).cpu().numpy()
            out[name] = a.view(np.uint32) if "codes" in name else a.view(np.uint16)
        return out
