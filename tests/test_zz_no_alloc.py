"""attn_decode_static: the attention call for callers that cannot allocate
device memory (a plugin that only receives input/output pointers, or a
serving loop that forbids allocation after start-up).  It runs the same
kernels as attn_decode with the library's static scratch array instead of a
caller workspace.  This file is named to be collected last; it must pass both
alone in a fresh process and after the other tests."""
import numpy as np
import pytest

import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 1e-2, 1e-3


@pytest.fixture(scope="module")
def kvq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_kv_attention_quant_gb300 as m
    from quantized_kv_attention_quant_gb300 import harness
    return m, harness


def _static_call(m, case, out):
    m.attn_decode_static(case.lay, case.caches.desc, case.wl.n_seqs, case.pos, case.max_pos, case.q, case.q_w,
                         out, 1)


def _static_status(m) -> int:
    word = np.full(1, 0xFFFFFFFF, np.uint32)      # pageable host memory: the copy is done on return
    m.kvq_static_status(word)
    torch.cuda.synchronize()
    return int(word[0])


def _device_memory():
    """(free device bytes, torch allocations so far): a cudaMalloc of the
    library moves the first, one through torch the second."""
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0], torch.cuda.memory_stats().get("allocation.all.allocated", 0)


@pytest.mark.parametrize("name,spec,filled,bits", [
    ("sliding-mixed-bits", W.LayerSpec(8, 2, 256, 512, 256, 1e4, False), [700, 40, 513], [4, 8, 4]),
    ("full-keqv", W.LayerSpec(16, 1, 512, 0, 128, 1e6, True), [2000, 65, 1], [4, 8, 4]),
])
def test_static_scratch_matches_workspace_call(kvq, name, spec, filled, bits):
    m, harness = kvq
    wl = W.DecodeWorkload(name, 91, spec, filled=filled, bits=bits)
    case = harness.DecodeCase(wl)            # fills the caches
    case.append()
    case.attend()                           # attn_decode with a torch-allocated workspace
    torch.cuda.synchronize()
    ref = case.out.cpu().numpy().copy()
    assert np.all(np.isfinite(ref))
    outs = [torch.full_like(case.out, float("nan")) for _ in range(3)]
    _static_call(m, case, outs[2])          # first use on this device: looks up the array, loads kernels
    assert _static_status(m) == 0
    before = _device_memory()
    for out in outs[:2]:                    # two calls in a row share the static scratch
        _static_call(m, case, out)
        torch.cuda.synchronize()
        assert _static_status(m) == 0
        got = out.cpu().numpy()
        d = np.abs(got.astype(np.float64) - ref)
        assert d.max() <= MAX_ABS and d.mean() <= MEAN_ABS, (d.max(), d.mean())
    assert _device_memory() == before, "a static call allocated device memory"


def test_static_scratch_rejects_oversized_call(kvq):
    m, _ = kvq
    lay = m.layer(16, 1, 512, 0, 128, 1e6, k_eq_v=True)
    n = 4096                                 # many rows: needs more than the static buffer
    assert m.attn_decode_workspace_bytes(lay, n, 1 << 15) > m.KVQ_STATIC_SCRATCH_BYTES
    with pytest.raises(m.KvqError) as e:
        m.attn_decode_static(lay, 1 << 20, n, 1 << 20, 1 << 15, 1 << 20, 1 << 20, 1 << 20, 1)
    assert e.value.status == m.KVQ_EWORKSPACE
