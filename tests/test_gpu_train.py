"""The training forward's stateless read on the GPU (kvq_train_kv_prep +
attn_train_forward, through the C ABI) against the float64 oracle: the plain
keys and values and the prepped q rows bit-exact, the outputs within max-abs
1e-2 and mean-abs 1e-3.  Layouts: a prefix shared by ragged branches (an
empty branch, one-row branches, branches longer than a 128-row tile), no
prefix, a single causal block; full and sliding layers with windows that cut
into the prefix, window 1 and a window longer than the sequence; head_dim
64..512 and 1..16 q heads per kv head; a KV-sharing layer reading its
donor's keys and values; the 42-layer stack's shapes at full size."""
import dataclasses

import numpy as np
import pytest

import oracle as O
import workloads as W
from oracle_ref import attn_errors, expect_train

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


def _spec(n_q, n_kv, D, window, rope_dims, theta=1e4, k_eq_v=False):
    return W.LayerSpec(n_q, n_kv, D, window, rope_dims, theta, k_eq_v)


def _bits(t):
    return t.cpu().numpy().view(np.uint16)


def verify_train(case, wl, layer_id=0, rows=None, kv=None):
    torch.cuda.synchronize()
    assert case.status_word() == 0
    k_hat, v_hat, q_hat, outs = expect_train(wl, layer_id, rows=rows, kv=kv)
    if case.donor:
        assert np.array_equal(_bits(case.k_hat), O.f64_to_bf16(k_hat))
        assert np.array_equal(_bits(case.v_hat), O.f64_to_bf16(v_hat))
    if case.q_prepped is not None:
        assert np.array_equal(_bits(case.q_prepped), O.f64_to_bf16(q_hat))
    out = case.out.cpu().numpy()
    worst_max, worst_mean = 0.0, 0.0
    for r, want in outs.items():
        mx, mn = attn_errors(out[r], want)
        worst_max, worst_mean = max(worst_max, mx), max(worst_mean, mn)
    assert worst_max <= MAX_ABS and worst_mean <= MEAN_ABS, (wl.name, worst_max, worst_mean)
    return k_hat, v_hat, worst_max


def check_train(harness, wl, layer_id=0, rows=None):
    case = harness.TrainCase(wl, keep_prepped=True, layer_id=layer_id)
    case.step()
    verify_train(case, wl, layer_id, rows)
    return case


TRAIN_CASES = {
    # a prefix shared by ragged branches on a sliding layer whose window cuts into the prefix
    "d256-sliding-prefix": (_spec(8, 2, 256, 64, 256), [200, 70, 1, 0, 150]),
    # full K = V layer, 16 q heads per kv head (8 rows per tile), partial RoPE
    "d512-keqv-full": (_spec(16, 1, 512, 0, 128, 1e6, True), [100, 40, 70]),
    # one causal block (the plain training read)
    "d128-gqa2-causal": (_spec(4, 2, 128, 0, 64), [333]),
    # no prefix: every branch alone
    "d64-gqa16-no-prefix": (_spec(32, 2, 64, 0, 64), [0, 90, 45]),
    # window 1: every row reads only itself
    "d64-mha-window1": (_spec(2, 2, 64, 1, 0), [20, 5]),
    # one q head per kv head (128-row tiles), a branch one row longer than a tile
    "d256-g1": (_spec(2, 2, 256, 0, 256), [300, 129]),
    # window longer than the sequence, 8 q heads per kv head
    "d128-g8-long-window": (_spec(16, 2, 128, 1000, 128), [64, 64, 63]),
    # the sliding window reaching back from a long branch into the prefix
    "d512-sliding-window-d512": (_spec(16, 1, 512, 96, 512), [150, 130]),
}


@pytest.mark.parametrize("name", sorted(TRAIN_CASES))
def test_train_small(kvq, name):
    _, harness = kvq
    spec, blocks = TRAIN_CASES[name]
    check_train(harness, W.TrainWorkload(name, 71, spec, blocks))


@pytest.mark.parametrize("name", ["d256-sliding-prefix", "d512-keqv-full", "d64-gqa16-no-prefix"])
def test_train_donor_forward_equals_separate_calls(kvq, name):
    """attn_train_donor_forward (the donor's K/V prep in the grid of the read's
    q prep) gives the bytes of kvq_train_kv_prep + attn_train_forward."""
    _, harness = kvq
    spec, blocks = TRAIN_CASES[name]
    wl = W.TrainWorkload("fused-" + name, 75, spec, blocks)
    a = harness.TrainCase(wl, keep_prepped=True, layer_id=5)
    b = harness.TrainCase(wl, keep_prepped=True, layer_id=5)
    a.step()
    b.step(fused=True)
    torch.cuda.synchronize()
    assert a.status_word() == b.status_word() == 0
    for x, y in ((a.out, b.out), (a.q_prepped, b.q_prepped), (a.k_hat, b.k_hat), (a.v_hat, b.v_hat)):
        assert torch.equal(x, y)
    verify_train(b, wl, 5)


def test_train_sharer_reads_donor_kv(kvq):
    """A KV-sharing layer (its own q rows and weights) reads the donor's plain
    keys and values."""
    _, harness = kvq
    wl = W.TrainWorkload("share", 72, _spec(8, 2, 256, 0, 256), [130, 60, 77])
    donor = harness.TrainCase(wl, keep_prepped=True, layer_id=3)
    donor.step()
    sharer = harness.TrainCase(wl, keep_prepped=True, kv=donor.kv, layer_id=9)
    sharer.step()
    k_hat, v_hat, _ = verify_train(donor, wl, 3)
    verify_train(sharer, wl, 9, kv=(k_hat, v_hat))


def test_train_bf16_output_is_rounded_f32(kvq):
    _, harness = kvq
    spec, blocks = TRAIN_CASES["d256-sliding-prefix"]
    wl = W.TrainWorkload("bf16", 73, spec, blocks)
    a = harness.TrainCase(wl)
    a.step()
    b = harness.TrainCase(wl, out_f32=False)
    b.step()
    torch.cuda.synchronize()
    f32 = a.out.cpu().numpy().astype(np.float64)
    assert np.array_equal(_bits(b.out), O.f64_to_bf16(O.rn_bf16(f32)))


def test_train_bad_layout_is_flagged(kvq):
    """Blocks whose offsets break the layout are skipped with the status bit;
    the valid prefix block is still read correctly."""
    m, harness = kvq
    spec = _spec(8, 2, 256, 0, 256)
    wl = W.TrainWorkload("bad", 74, spec, [50, 50])
    case = harness.TrainCase(wl, keep_prepped=True)
    case.prep_kv()
    case.offs = torch.tensor([0, 50, 40], dtype=torch.int32, device="cuda")     # block 1 runs backwards
    case.out.fill_(float("nan"))
    case.attend()
    torch.cuda.synchronize()
    assert case.status_word() & m.KVQ_STATUS_SEQ_SKIPPED
    _, _, _, outs = expect_train(W.TrainWorkload("bad", 74, spec, [50, 50]), rows=range(50))
    out = case.out.cpu().numpy()
    for r, want in outs.items():
        assert attn_errors(out[r], want)[0] <= MAX_ABS
    assert np.isnan(out[50:]).all()


@pytest.mark.parametrize("kind", ["sliding", "full"])
def test_workload_train_prefix_shared(kvq, kind):
    """The stack's two layer shapes over the measured layout (prefix 1024,
    four branches of 256): every prepped row bit-exact, outputs on sampled
    rows (the first and last rows of every block and tile edges)."""
    _, harness = kvq
    sliding, full = W.workload_train_prefix_shared()
    wl = sliding if kind == "sliding" else full
    off = wl.offsets()
    rows = sorted({int(x) for b in range(len(off) - 1) if off[b + 1] > off[b]
                   for x in (off[b], off[b] + 1, off[b] + 127, off[b] + 128, off[b + 1] - 1)})
    check_train(harness, wl, layer_id=5 if kind == "full" else 0, rows=rows)


@pytest.mark.parametrize("blocks", [[1], [0, 1], [37, 0, 0], [5, 1, 1, 1]])
def test_train_tiny_layouts(kvq, blocks):
    """One row; a branch of one row and no prefix; a prefix whose branches are
    all empty; one-row branches (D512 K = V and D128 window 3)."""
    _, harness = kvq
    for spec in (_spec(16, 1, 512, 0, 128, 1e6, True), _spec(4, 2, 128, 3, 128)):
        check_train(harness, W.TrainWorkload("tiny", 75, spec, list(blocks)))


def test_train_grid_larger_than_blocks(kvq):
    """max_block_rows above every block (extra row tiles return at once)."""
    _, harness = kvq
    spec, blocks = TRAIN_CASES["d256-sliding-prefix"]
    wl = W.TrainWorkload("grid", 76, spec, blocks)
    case = harness.TrainCase(wl, keep_prepped=True)
    case.max_rows = wl.n_rows
    case.step()
    verify_train(case, wl)
