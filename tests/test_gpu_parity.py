"""GPU path vs the float64 oracle, element by element, through the C ABI.

Bars (from the statement of the method): the prepped bf16 rows and the packed
codes / scales / biases bit-exact; attention outputs (fp32) within max-abs
1e-2 and mean-abs 1e-3 of the oracle.  Sizes span several 64-key tiles with a
ragged tail; the edge cases cover the first token, window 1, window larger
than the history, ring wrap-around, rope_dims 0 / partial / full, GQA ratios
1..16, head_dim 64..512, 4- and 8-bit caches mixed across sequences.
"""
import dataclasses

import numpy as np
import pytest

import oracle as O
import workloads as W
from oracle_ref import (EDGE_BITS, EDGE_SPEC, attn_errors, compare_cache, edge_inputs, expect_decode,
                        expect_edge, expect_prefill, expect_shared, ring_slots)

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


def check_decode(harness, wl, seqs=None, check_fill=True):
    case = harness.DecodeCase(wl, keep_prepped=True, keep_fill=check_fill)
    case.step()
    torch.cuda.synchronize()
    return case, verify_decode(case, wl, seqs, check_fill)


def verify_decode(case, wl, seqs=None, check_fill=True):
    """The stepped case against the oracle: prepped rows and cache bytes
    bit-exact, outputs within the tolerance.  Returns the worst errors."""
    assert case.status_word() == 0
    out = case.out.cpu().numpy()
    qp = case.q_prepped.cpu().numpy().view(np.uint16)
    kvp = case.kv_prepped.cpu().numpy().view(np.uint16)
    worst = (0.0, 0.0)
    for s in (range(wl.n_seqs) if seqs is None else seqs):
        e = expect_decode(wl, s)
        if check_fill and len(e.fill_positions):
            got = case.fill_prepped[s]
            assert np.array_equal(got[0], O.f64_to_bf16(e.fill_k_hat)), f"seq {s}: fill k prep"
            assert np.array_equal(got[1], O.f64_to_bf16(e.fill_v_hat)), f"seq {s}: fill v prep"
        assert np.array_equal(qp[s], O.f64_to_bf16(e.q_hat[0])), f"seq {s}: q prep"
        assert np.array_equal(kvp[0, s], O.f64_to_bf16(e.k_hat[0])), f"seq {s}: k prep"
        assert np.array_equal(kvp[1, s], O.f64_to_bf16(e.v_hat[0])), f"seq {s}: v prep"
        rows = case.caches.host_rows(s, ring_slots(e.resident, wl.capacity(s)))
        assert compare_cache(rows, e.cache, e.resident) == 0, f"seq {s}: cache bytes"
        mx, mean = attn_errors(out[s], e.out[0])
        assert mx <= MAX_ABS and mean <= MEAN_ABS, f"seq {s}: max {mx} mean {mean}"
        worst = (max(worst[0], mx), max(worst[1], mean))
    return worst


DECODE_CASES = {
    # name: (spec, filled per seq, bits per seq)
    "sliding-ring-wrap": (_spec(8, 2, 256, 100, 256), [300, 99, 5], [4, 8, 4]),
    "full-keqv-partial-rope": (_spec(16, 1, 512, 0, 128, 1e6, True), [0, 1, 63, 64, 65, 700], [4, 8, 4, 8, 4, 8]),
    "window-1": (_spec(8, 2, 256, 1, 256), [0, 37, 200], [4, 8, 8]),
    "window-over-history": (_spec(8, 2, 256, 4096, 256), [200, 1], [8, 4]),
    "mha-no-rope-d128": (_spec(4, 4, 128, 0, 0), [129, 3], [4, 8]),
    "d64-full-rope": (_spec(2, 1, 64, 0, 64), [80, 64], [8, 4]),
    "gqa8-d256": (_spec(8, 1, 256, 0, 64, 1e6), [190], [4]),
    "gqa1-d512-window": (_spec(2, 2, 512, 64, 512), [130, 64], [8, 4]),
    # G = 3 (not a power of two), a large eps and a single rotated pair
    "gqa3-eps-half-rope2": (W.LayerSpec(6, 2, 256, 0, 2, 1e4, False, rms_eps=0.5), [100, 7], [4, 8]),
    # 16 q heads per kv head at head_dim 64 (one warp per CTA)
    "d64-gqa16": (_spec(32, 2, 64, 0, 64), [200, 5, 70], [4, 8, 4]),
}


@pytest.mark.parametrize("name", sorted(DECODE_CASES))
def test_decode_small(kvq, name):
    _, harness = kvq
    spec, filled, bits = DECODE_CASES[name]
    wl = W.DecodeWorkload(name, 77, spec, filled=filled, bits=bits)
    _, worst = check_decode(harness, wl)
    print(name, "worst", worst)


# Batches whose longest row spans more than one 48-tile chunk take the
# stream-K schedule: equal tile ranges per CTA across (row, kv head) units,
# rows inside one range written directly, the others merged from pieces.
STREAM_K_CASES = {
    "sk-ragged-d512-keqv": (_spec(16, 1, 512, 0, 128, 1e6, True),
                            [3100, 20, 500, 4000, 64, 3500, 0, 700], [4, 8, 8, 4, 4, 8, 4, 8]),
    "sk-ragged-d256-full": (_spec(8, 2, 256, 0, 256), [3300, 100, 2000, 3999, 63], [8, 4, 4, 8, 8]),
    "sk-equal-rows-d512": (_spec(16, 1, 512, 0, 128, 1e6, True), [3500] * 4, [4, 8, 4, 8]),
    "sk-gqa8-d128": (_spec(8, 1, 128, 0, 128), [5000, 3072, 3073, 17], [8, 4, 8, 4]),
    "sk-gqa16-d64": (_spec(16, 1, 64, 0, 32), [4000, 3300, 20, 3100], [8, 4, 4, 8]),
}


@pytest.mark.parametrize("name", sorted(STREAM_K_CASES))
def test_decode_stream_k(kvq, name):
    _, harness = kvq
    spec, filled, bits = STREAM_K_CASES[name]
    wl = W.DecodeWorkload(name, 78, spec, filled=filled, bits=bits)
    _, worst = check_decode(harness, wl, check_fill=False)
    print(name, "worst", worst)


def test_stream_k_bf16_output_is_rounded_f32(kvq):
    """bf16 outputs of the stream-K schedule (rows finished inside one CTA are
    written by the attention kernel, the others by the merge) are exactly the
    rounded fp32 outputs."""
    _, harness = kvq
    spec, filled, bits = STREAM_K_CASES["sk-ragged-d512-keqv"]
    wl = W.DecodeWorkload("sk-bf16", 79, spec, filled=filled, bits=bits)
    a = harness.DecodeCase(wl)
    a.step()
    b = harness.DecodeCase(wl, out_f32=False)
    b.step()
    torch.cuda.synchronize()
    f32 = a.out.cpu().numpy()
    bf = b.out.cpu().numpy().view(np.uint16)
    assert np.array_equal(bf, O.f64_to_bf16(O.rn_bf16(f32.astype(np.float64))))


def test_many_rows_take_fixed_chunks(kvq):
    """Over 1024 rows per call the decode falls back from stream-K to fixed
    48-tile chunks; rows longer than one chunk still merge correctly."""
    _, harness = kvq
    spec = _spec(2, 1, 64, 0, 64)
    rng = np.random.default_rng(84)
    filled = [int(x) for x in rng.integers(0, 200, size=1030)]
    for s, n in ((3, 3100), (517, 5000), (1029, 3072)):
        filled[s] = n
    bits = [int(b) for b in rng.choice([4, 8], size=1030)]
    wl = W.DecodeWorkload("many-rows", 84, spec, filled=filled, bits=bits)
    _, worst = check_decode(harness, wl, seqs=[0, 3, 4, 517, 700, 1029], check_fill=False)
    print("many-rows worst", worst)


# attn_decode_append: one call for a donor's append and read, bit-equal to
# kv_quant_append + attn_decode.  Cases: a window ring that is exactly the
# window (row 611 of a 512-slot ring sees keys 100..611, whose first and last
# tiles share a ring tile: the first is copied early, the last after the
# append), fresh caches (position 0: the first tile is the new one), ragged
# stream-K rows, GQA 16 at D64, a rotated layer, a skipped sequence.
FUSED_CASES = {
    "sliding-ring-exact": (_spec(8, 2, 256, 512, 256), [611, 512, 511, 0, 1000, 63], [4, 8, 8, 4, 4, 8]),
    "full-keqv-stream-k": STREAM_K_CASES["sk-ragged-d512-keqv"],
    "d64-gqa16": DECODE_CASES["d64-gqa16"],
    "rot-full-keqv": (dataclasses.replace(_spec(16, 1, 512, 0, 128, 1e6, True), kv_rotation=True),
                      [900, 0, 64, 2000], [4, 8, 8, 4]),
}


def _fused_pair(harness, wl):
    """The same step twice on identical caches: separate calls, then the fused
    call.  Returns the two cases after the steps."""
    a = harness.DecodeCase(wl, keep_prepped=True)
    b = harness.DecodeCase(wl, keep_prepped=True)
    a.step()
    b.append_attend()
    torch.cuda.synchronize()
    return a, b


@pytest.mark.parametrize("name", sorted(FUSED_CASES))
def test_decode_append_equals_separate_calls(kvq, name):
    _, harness = kvq
    spec, filled, bits = FUSED_CASES[name]
    wl = W.DecodeWorkload("fused-" + name, 96, spec, filled=filled, bits=bits)
    a, b = _fused_pair(harness, wl)
    assert a.status_word() == b.status_word() == 0
    for x, y in ((a.out, b.out), (a.q_prepped, b.q_prepped), (a.kv_prepped, b.kv_prepped)):
        assert torch.equal(x, y)
    for s in range(wl.n_seqs):
        slots = ring_slots(wl.filled[s] + 1, wl.capacity(s))
        assert np.array_equal(a.caches.host_rows(s, slots)["k_codes"], b.caches.host_rows(s, slots)["k_codes"])
    worst = verify_decode(b, wl, check_fill=False)
    print(name, "worst", worst)


def test_profile_events_time_the_attention_kernel(kvq):
    """kvq_profile_next_read: the next call records the event pair around its
    attention kernel (inside the call's own span); its outputs are those of a
    plain call; the call after it records nothing."""
    m, harness = kvq
    spec, filled, bits = STREAM_K_CASES["sk-ragged-d512-keqv"]
    wl = W.DecodeWorkload("profile", 95, spec, filled=filled, bits=bits)
    case = harness.DecodeCase(wl)
    case.step()
    torch.cuda.synchronize()
    want = case.out.clone()
    k0, k1, c0, c1 = (torch.cuda.Event(enable_timing=True) for _ in range(4))
    k0.record()
    k1.record()
    torch.cuda.synchronize()
    c0.record()
    m.kvq_profile_next_read(k0, k1)
    case.attend()
    c1.record()
    torch.cuda.synchronize()
    kern, call = k0.elapsed_time(k1), c0.elapsed_time(c1)
    assert 0 < kern <= call
    assert torch.equal(case.out, want)
    case.attend()                     # the pair is spent: the kernel's events stay as they were
    torch.cuda.synchronize()
    assert k0.elapsed_time(k1) == kern
    with pytest.raises(m.KvqError):
        m.kvq_profile_next_read(k0, None)


def test_decode_append_skips_a_bad_sequence(kvq):
    """A sequence with an invalid descriptor inside a fused call: nothing of
    it is written, its output is NaN, the status word says so, and the other
    sequences are as the oracle has them."""
    _, harness = kvq
    spec = _spec(8, 2, 256, 512, 256)
    wl = W.DecodeWorkload("fused-bad", 97, spec, filled=[300, 40, 700], bits=[8, 4, 4])
    c = harness.DecodeCase(wl, keep_prepped=True)
    torch.cuda.synchronize()
    before = c.caches.seqs[1]["k_codes"].clone()
    bad = c.caches.desc.cpu().numpy().copy()
    bad[56 + 48:56 + 52] = np.frombuffer(np.int32(5).tobytes(), np.uint8)      # seq 1: bits = 5
    c.caches.desc.copy_(torch.from_numpy(bad))
    c.append_attend()
    torch.cuda.synchronize()
    assert c.status_word() & (1 << 2)
    out = c.out.cpu().numpy()
    assert np.all(np.isnan(out[1]))
    assert torch.equal(before, c.caches.seqs[1]["k_codes"])
    good = harness.DecodeCase(wl, keep_prepped=True)
    good.step()
    torch.cuda.synchronize()
    assert torch.equal(c.out[[0, 2]], good.out[[0, 2]])


# the deferred TurboQuant read (rotated K/V, q rotated, output un-rotated):
# fixed chunks, stream-K with rows merged and rows written by one CTA, a
# window layer and a prompt chunk (the row path), 4- and 8-bit caches
ROT = dict(kv_rotation=True)
ROT_DECODE_CASES = {
    "rot-full-keqv-short": (_spec(16, 1, 512, 0, 128, 1e6, True), [0, 63, 64, 900, 2000], [4, 8, 8, 4, 8]),
    "rot-full-keqv-stream-k": (_spec(16, 1, 512, 0, 128, 1e6, True), [3300, 20, 5000, 4100, 700, 64],
                               [8, 4, 4, 8, 8, 4]),
    "rot-sliding-d256": (_spec(8, 2, 256, 512, 256), [600, 40, 1500], [4, 8, 8]),
    "rot-d64-gqa16": (_spec(32, 2, 64, 0, 64), [300, 9], [8, 4]),
}


@pytest.mark.parametrize("name", sorted(ROT_DECODE_CASES))
def test_rotated_decode(kvq, name):
    """Rotated rows (q, k, v and every cached row) bit-exact, caches bit-exact,
    outputs within the tolerance of the oracle's rotated read."""
    _, harness = kvq
    spec, filled, bits = ROT_DECODE_CASES[name]
    wl = W.DecodeWorkload(name, 96, dataclasses.replace(spec, **ROT), filled=filled, bits=bits)
    _, worst = check_decode(harness, wl)
    print(name, "worst", worst)


def test_rotated_prompt_chunks_and_bf16_output(kvq):
    """Prompt chunks and verify windows on rotated layers (the row path, which
    the merge un-rotates), and the bf16 output of a rotated read is the
    rounded fp32 one."""
    _, harness = kvq
    wl = W.PrefillWorkload("rot-chunk-d512", 97, dataclasses.replace(_spec(16, 1, 512, 0, 128, 1e6, True), **ROT),
                           filled=[130, 5], chunk=[40, 9], bits=[4, 8])
    check_prefill(harness, wl)
    wl = W.PrefillWorkload("rot-chunk-d256", 97, dataclasses.replace(_spec(8, 2, 256, 64, 256), **ROT),
                           filled=[150, 0], chunk=[30, 12], bits=[8, 4])
    check_prefill(harness, wl)
    spec, filled, bits = ROT_DECODE_CASES["rot-full-keqv-stream-k"]
    wl = W.DecodeWorkload("rot-bf16", 98, dataclasses.replace(spec, **ROT), filled=filled, bits=bits)
    a = harness.DecodeCase(wl)
    a.step()
    b = harness.DecodeCase(wl, out_f32=False)
    b.step()
    torch.cuda.synchronize()
    f32 = a.out.cpu().numpy()
    assert np.array_equal(b.out.cpu().numpy().view(np.uint16), O.f64_to_bf16(O.rn_bf16(f32.astype(np.float64))))


def test_stream_k_bad_descriptor_is_nan(kvq):
    """A skipped sequence inside a stream-K batch: NaN rows, status bit set,
    the other rows unaffected."""
    _, harness = kvq
    spec = _spec(16, 1, 512, 0, 128, 1e6, True)
    wl = W.DecodeWorkload("sk-bad", 83, spec, filled=[3200, 3300, 100], bits=[8, 4, 8])
    case = harness.DecodeCase(wl)
    case.step()
    torch.cuda.synchronize()
    good = case.out.cpu().numpy().copy()
    raw = case.caches.desc.cpu().numpy().copy()
    bad = raw.copy()
    bad[56 + 48:56 + 52] = np.frombuffer(np.int32(5).tobytes(), np.uint8)      # seq 1: bits = 5
    case.caches.desc.copy_(torch.from_numpy(bad))
    case.attend()
    torch.cuda.synchronize()
    out = case.out.cpu().numpy()
    assert np.all(np.isnan(out[1]))
    # the other rows' tiles are split at other points now: equal up to rounding
    assert np.allclose(out[0], good[0], atol=1e-4) and np.allclose(out[2], good[2], atol=1e-4)
    assert case.status_word() & (1 << 2)


def test_rope_frequencies_on_this_host():
    """The frequency table both sides derive from the platform pow is the
    nearest-double table of tests/golden/rope_freqs.txt on the machine that
    runs the GPU tests too (its libm may differ from the one the CPU pins ran
    on)."""
    from test_oracle_pins import read_rope_freqs
    for (theta, D), want in read_rope_freqs().items():
        assert [float(x) for x in O.rope_inv_freq(theta, D, D)] == want, (theta, D)


def test_bounded_wait_gives_up(kvq):
    """Failure detection without a fault: the kernels' bounded wait on an
    mbarrier that nothing completes gives up, sets the timeout bit, and the
    context stays usable for the next call."""
    m, harness = kvq
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.kvq_selftest_wait_timeout(status, 5_000_000)        # 5 ms
    torch.cuda.synchronize()
    assert int(status.item()) & (1 << 1)
    spec, filled, bits = DECODE_CASES["window-1"]
    check_decode(harness, W.DecodeWorkload("after-timeout", 77, spec, filled=filled, bits=bits))


def test_decode_bf16_output_is_rounded_f32(kvq):
    _, harness = kvq
    spec, filled, bits = DECODE_CASES["sliding-ring-wrap"]
    wl = W.DecodeWorkload("bf16out", 78, spec, filled=filled, bits=bits)
    a = harness.DecodeCase(wl)
    a.step()
    b = harness.DecodeCase(wl, out_f32=False)
    b.step()
    torch.cuda.synchronize()
    f32 = a.out.cpu().numpy()
    bf = b.out.cpu().numpy().view(np.uint16)
    want = O.f64_to_bf16(O.rn_bf16(f32.astype(np.float64)))
    assert np.array_equal(bf, want)


def check_prefill(harness, wl, seqs=None, rows=None, nan_rows=None):
    case = harness.PrefillCase(wl, keep_prepped=True)
    case.step()
    torch.cuda.synchronize()
    return case, verify_prefill(case, wl, seqs, rows, nan_rows)


def verify_prefill(case, wl, seqs=None, rows=None, nan_rows=None):
    out = case.out.cpu().numpy()
    qp = case.q_prepped.cpu().numpy().view(np.uint16)
    kvp = case.kv_prepped.cpu().numpy().view(np.uint16)
    offs = np.concatenate([[0], np.cumsum(wl.chunk)])
    worst = (0.0, 0.0)
    for s in (range(wl.n_seqs) if seqs is None else seqs):
        e = expect_prefill(wl, s, rows=rows)
        r0, r1 = offs[s], offs[s + 1]
        assert np.array_equal(qp[r0:r1], O.f64_to_bf16(e.q_hat)), f"seq {s}: q prep"
        assert np.array_equal(kvp[0, r0:r1], O.f64_to_bf16(e.k_hat)), f"seq {s}: k prep"
        assert np.array_equal(kvp[1, r0:r1], O.f64_to_bf16(e.v_hat)), f"seq {s}: v prep"
        cache_rows = case.caches.host_rows(s, ring_slots(e.resident, wl.capacity(s)))
        assert compare_cache(cache_rows, e.cache, e.resident) == 0, f"seq {s}: cache bytes"
        for t, want in e.out.items():
            got = out[r0 + t]
            if nan_rows is not None and t in nan_rows.get(s, ()):
                assert np.all(np.isnan(got)), f"seq {s} row {t}: expected NaN"
                continue
            mx, mean = attn_errors(got, want)
            assert mx <= MAX_ABS and mean <= MEAN_ABS, f"seq {s} row {t}: max {mx} mean {mean}"
            worst = (max(worst[0], mx), max(worst[1], mean))
    return worst


def test_prefill_small_sliding(kvq):
    _, harness = kvq
    spec = _spec(8, 2, 256, 64, 256)
    wl = W.PrefillWorkload("prefill-sliding", 79, spec, filled=[150, 0], chunk=[100, 37], bits=[8, 4])
    _, worst = check_prefill(harness, wl)
    print("worst", worst)


def test_prefill_small_full_keqv(kvq):
    _, harness = kvq
    spec = _spec(16, 1, 512, 0, 128, 1e6, True)
    wl = W.PrefillWorkload("prefill-full", 80, spec, filled=[130, 5], chunk=[70, 9], bits=[4, 8])
    check_prefill(harness, wl)


def test_prefill_rows_beyond_ring_are_nan(kvq):
    """A chunk longer than its ring keeps only the newest `capacity` rows; rows
    whose window reaches an overwritten key are reported as NaN."""
    _, harness = kvq
    spec = _spec(4, 1, 128, 64, 128)
    wl = W.PrefillWorkload("prefill-overflow", 81, spec, filled=[10], chunk=[300], bits=[4])
    cap = wl.capacity(0)                      # ring for chunk 300 = 384 slots: no overflow
    assert cap >= 300 + 64 - 1
    wl2 = dataclasses.replace(wl)
    wl2.capacity = lambda s: 192              # force a too-small ring
    wl2.cached_positions = lambda s: np.arange(0, 10)
    newest = 10 + 300 - 1
    valid_from = newest - 192 + 1 + 63 - 10   # row index whose window start fits
    nan_rows = {0: set(range(0, valid_from))}
    check_prefill(harness, wl2, rows=[0, valid_from - 1, valid_from, 299], nan_rows=nan_rows)


def test_bad_descriptor_is_skipped(kvq):
    """A descriptor with an unsupported width or a misaligned pointer is
    skipped by the kernels: nothing written, NaN outputs, status bit set."""
    m, harness = kvq
    spec = _spec(8, 2, 256, 0, 256)
    wl = W.DecodeWorkload("bad", 82, spec, filled=[70, 70], bits=[4, 4])
    case = harness.DecodeCase(wl)
    torch.cuda.synchronize()
    raw = case.caches.desc.cpu().numpy().copy()
    before = case.caches.seqs[1]["k_codes"].clone()
    bad = raw.copy()
    bad[56 + 48:56 + 52] = np.frombuffer(np.int32(5).tobytes(), np.uint8)      # bits = 5
    case.caches.desc.copy_(torch.from_numpy(bad))
    case.step()
    torch.cuda.synchronize()
    out = case.out.cpu().numpy()
    assert np.all(np.isnan(out[1])) and np.all(np.isfinite(out[0]))
    assert case.status_word() & (1 << 2)
    assert torch.equal(before, case.caches.seqs[1]["k_codes"])
    # misaligned scale pointer (still inside its allocation)
    mis = raw.copy()
    p = int(np.frombuffer(mis[56 + 16:56 + 24].tobytes(), np.uint64)[0]) + 2
    mis[56 + 16:56 + 24] = np.frombuffer(np.uint64(p).tobytes(), np.uint8)
    case.caches.desc.copy_(torch.from_numpy(mis))
    case.attend()
    torch.cuda.synchronize()
    assert np.all(np.isnan(case.out.cpu().numpy()[1]))


def test_largest_positions(kvq):
    """Positions up to 2^24 - 1, the largest the calls accept, on window
    layers (the ring holds only the window, so the caches stay small): decode
    at D256 with full RoPE and at D512 with partial RoPE and K = V, and a
    prompt chunk ending at 2^24 - 2.  Some positions put cos or sin of a
    rotary angle next to zero, where the angle has to be formed without
    rounding to give the right bf16 row."""
    _, harness = kvq
    P = 2 ** 24 - 1
    wl = W.DecodeWorkload("pos-max-d256", 87, _spec(8, 2, 256, 64, 256),
                          filled=[P, P - 1, 11039086, 14207257, 2 ** 23], bits=[4, 8, 8, 4, 8])
    check_decode(harness, wl)
    wl = W.DecodeWorkload("pos-max-d512-keqv", 88, _spec(16, 1, 512, 64, 128, 1e6, True),
                          filled=[P, 11311958, 10761476], bits=[8, 4, 8])
    check_decode(harness, wl)
    wl = W.PrefillWorkload("pos-max-chunk", 89, _spec(8, 2, 256, 64, 256),
                           filled=[P - 40, 11039080], chunk=[40, 17], bits=[8, 4])
    check_prefill(harness, wl)


def test_quantizer_edge_rows(kvq):
    """Hand-designed groups (an fp32-quotient midpoint, exact ties, a constant
    group, a -0 minimum, a bf16 scale that is not (max - min) / (2^b - 1), a
    nearly constant and an all-negative group, a bf16-subnormal scale whose
    float32 reciprocal overflows) appended as one prompt chunk
    into a 4-bit and an 8-bit cache: prepped rows and cache bytes bit-exact
    with the oracle, the designed codes read back from the GPU cache, then the
    prompt path (every row) and the decode path (the last row) within the
    tolerance."""
    m, harness = kvq
    from quantized_kv_attention_quant_gb300.cache import LayerCaches
    names, k, v, q, w = edge_inputs()
    n, D, dev = len(names), EDGE_SPEC.head_dim, "cuda"
    ns = len(EDGE_BITS)
    lay = harness.kvq_layer(EDGE_SPEC)
    caches = LayerCaches(1, D, list(EDGE_BITS), [W.TILE_KEYS] * ns, dev)
    w_d = harness.dev_bits(w, dev)
    k_d = harness.dev_bits(np.concatenate([k] * ns), dev)
    v_d = harness.dev_bits(np.concatenate([v] * ns), dev)
    q_d = harness.dev_bits(np.concatenate([q] * ns), dev)
    offs = harness.dev_i32(np.arange(ns + 1) * n, dev)
    start = harness.dev_i32([0] * ns, dev)
    kvp = torch.empty((2, ns * n, 1, D), dtype=torch.int16, device=dev)
    m.kv_quant_append(lay, caches.desc, ns, offs, start, ns * n, k_d, v_d, w_d, kvp)
    ws_bytes = m.attn_prefill_workspace_bytes(lay, ns, ns * n, n)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty((ns * n, EDGE_SPEC.n_q_heads, D), dtype=torch.float32, device=dev)
    m.attn_prefill_chunk(lay, caches.desc, ns, offs, start, ns * n, n, q_d, w_d, out, 1, None, ws, ws_bytes)
    pos = harness.dev_i32([n - 1] * ns, dev)
    q_last = harness.dev_bits(np.stack([q[n - 1]] * ns), dev)
    wsd_bytes = m.attn_decode_workspace_bytes(lay, ns, n - 1)
    wsd = torch.empty(wsd_bytes, dtype=torch.uint8, device=dev)
    out_d = torch.empty((ns, EDGE_SPEC.n_q_heads, D), dtype=torch.float32, device=dev)
    m.attn_decode(lay, caches.desc, ns, pos, n - 1, q_last, w_d, out_d, 1, None, wsd, wsd_bytes)
    torch.cuda.synchronize()
    assert int(ws[:4].cpu().numpy().view(np.uint32)[0]) == 0
    assert int(wsd[:4].cpu().numpy().view(np.uint32)[0]) == 0
    got_kv = kvp.cpu().numpy().view(np.uint16)
    got = out.cpu().numpy()
    got_d = out_d.cpu().numpy()
    for s, bits in enumerate(EDGE_BITS):
        e = expect_edge(bits)
        r = slice(s * n, (s + 1) * n)
        assert np.array_equal(got_kv[0, r], k) and np.array_equal(got_kv[1, r], v), f"{bits}-bit: prep"
        assert np.array_equal(got_kv[0, r], O.f64_to_bf16(e.k_hat)), f"{bits}-bit: k prep"
        rows = caches.host_rows(s, np.arange(n))
        assert compare_cache(rows, e.cache, np.arange(n)) == 0, f"{bits}-bit: cache bytes"
        # the designed codes, unpacked from the GPU's own words
        tie = names.index(f"fp32-quotient-tie-{bits}")
        c = O.unpack(rows["k_codes"][0, tie], bits)
        assert (c[0], c[1], c[2]) == ((0, 15, 0) if bits == 4 else (0, 254, 0))
        assert rows["k_biases"][0, names.index("negative-zero-min"), 0] == 0x0000
        assert rows["k_scales"][0, names.index("constant"), 0] == 0
        sub = names.index("subnormal-scale")
        c = O.unpack(rows["k_codes"][0, sub], bits)
        assert tuple(c[:4]) == ((0, 15, 6, 2) if bits == 4 else (0, 255, 100, 37))
        assert rows["k_scales"][0, sub, 0] == (0x0011 if bits == 4 else 0x0001)
        for t in range(n):
            mx, mean = attn_errors(got[s * n + t], e.out[t])
            assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{bits}-bit row {t} ({names[t]}): max {mx} mean {mean}"
        mx, mean = attn_errors(got_d[s], e.out[n - 1])
        assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{bits}-bit decode: max {mx} mean {mean}"


# ----------------------------------------------------------------------------
# the measured workloads at full size (sampled sequences where the oracle
# would take long)
# ----------------------------------------------------------------------------

def test_workload_tiny(kvq):
    check_decode(kvq[1], W.workload_tiny_decode())


def test_workload_sliding16(kvq):
    check_decode(kvq[1], W.workload_sliding_decode_b16(), seqs=[0, 7, 8, 15])


def test_workload_full32k(kvq):
    check_decode(kvq[1], W.workload_full_keqv_decode(), seqs=[3], check_fill=False)


def test_workload_prefill(kvq):
    check_prefill(kvq[1], W.workload_prefill_chunk(), seqs=[2], rows=[0, 1, 255, 511])


def test_workload_prefill_full(kvq):
    """The head_dim-512 prompt chunk at full size (the row path)."""
    check_prefill(kvq[1], W.workload_prefill_full(), seqs=[1], rows=[0, 1, 255, 511])


# layers of the 42-layer step compared with the oracle: full donors with an
# 8-bit (23) and a 4-bit (11) cache, the full sharer 41 (reads 23), the
# sliding donor 22 and the sliding sharer 24 (reads 22)
STACK_LAYERS = (11, 22, 23, 24, 41)


def test_workload_stack42(kvq):
    """The 42-layer KV-shared decode step at full size, as the bench runs it:
    64 ragged sequences of 1,798 .. 32,737 cached tokens, donors 0..23 append
    and attend (one attn_decode_append call each), sharers 24..41 attend the
    donor's cache without appending.  The
    full layers take the stream-K schedule over 64 rows (8-bit on donor 23 and
    its sharers).  On sampled sequences (every one of at least 32,000 keys, the
    shortest and the one nearest the mean length) of the listed layers: the
    prepped q rows and the new K/V rows bit-exact, every resident cache row of
    the donors bit-exact (codes, scales, biases), outputs within the tolerance."""
    _, harness = kvq
    wl = W.workload_stack_decode()
    assert (wl.donor_bits[23], wl.donor_bits[11], wl.donor_bits[22]) == (8, 4, 8)
    case = harness.StackCase(wl, inspect=STACK_LAYERS)
    case.step()
    torch.cuda.synchronize()
    L = np.asarray(wl.lengths)
    seqs = sorted(set(np.flatnonzero(L >= 32000).tolist())
                  | {int(np.argmin(L)), int(np.argmin(np.abs(L - L.mean())))})
    assert len(seqs) >= 5
    donors = {}
    worst = {}
    for i in STACK_LAYERS:
        _, d, lc = case.layers[i]
        assert lc.status_word() == 0, f"layer {i}: status"
        view = wl.decode_view(i)
        out = lc.out.cpu().numpy()
        qp = lc.q_prepped.cpu().numpy().view(np.uint16)
        kvp = lc.kv_prepped.cpu().numpy().view(np.uint16) if i == d else None
        for s in seqs:
            if (d, s) not in donors:
                donors[(d, s)] = expect_decode(view, s)
            e = donors[(d, s)]
            if i == d:
                q_hat, want = e.q_hat[0], e.out[0]
                assert np.array_equal(kvp[0, s], O.f64_to_bf16(e.k_hat[0])), f"layer {i} seq {s}: k prep"
                assert np.array_equal(kvp[1, s], O.f64_to_bf16(e.v_hat[0])), f"layer {i} seq {s}: v prep"
                rows = lc.caches.host_rows(s, ring_slots(e.resident, view.capacity(s)))
                assert compare_cache(rows, e.cache, e.resident) == 0, f"layer {i} seq {s}: cache bytes"
            else:
                q_hat, want = expect_shared(e, view, i, s)
            assert np.array_equal(qp[s], O.f64_to_bf16(q_hat)), f"layer {i} seq {s}: q prep"
            mx, mean = attn_errors(out[s], want)
            assert mx <= MAX_ABS and mean <= MEAN_ABS, f"layer {i} seq {s}: max {mx} mean {mean}"
            w = worst.get(i, (0.0, 0.0))
            worst[i] = (max(w[0], mx), max(w[1], mean))
    print("stack42 worst per layer", worst)


def test_stream_k_64_long_8bit_rows(kvq):
    """Stream-K over 64 rows of a head_dim-512 K = V layer with 8-bit caches,
    eight of them at 32,000 keys or more and the rest ragged: every CTA range
    crosses units, pieces of the long rows are merged from many CTAs.  Checked
    on the long rows, the shortest and two others."""
    _, harness = kvq
    rng = np.random.default_rng(94)
    filled = [int(x) for x in rng.integers(100, 24000, size=64)]
    for s in (0, 9, 21, 30, 31, 47, 58, 63):
        filled[s] = 32000 + 97 * s
    wl = W.DecodeWorkload("sk-64-long-8bit", 94, W.FULL_KEQV, filled=filled, bits=[8] * 64)
    seqs = [0, 9, 21, 30, 31, 47, 58, 63, int(np.argmin(filled)), 5, 40]
    _, worst = check_decode(harness, wl, seqs=sorted(set(seqs)), check_fill=False)
    print("sk-64-long-8bit worst", worst)


def test_workspace_contents_do_not_matter(kvq):
    """The workspace is scratch: NaN garbage left in it by earlier use must not
    reach the output (splits that read no keys write no o partial)."""
    _, harness = kvq
    spec, filled, bits = DECODE_CASES["sliding-ring-wrap"]
    wl = W.DecodeWorkload("ws-garbage", 83, spec, filled=filled, bits=bits)
    case = harness.DecodeCase(wl)
    case.step()
    torch.cuda.synchronize()
    ref = case.out.cpu().numpy().copy()
    case.ws.fill_(0xFF)                      # NaN bit patterns everywhere
    case.attend()
    torch.cuda.synchronize()
    assert np.array_equal(case.out.cpu().numpy(), ref)


def test_verify_windows(kvq):
    """Short windows of 2..64 query rows per sequence (speculative verify):
    the same call as a prompt chunk, on the tensor-core path (D256, G 4, a
    sequence of more than 16 rows), on the row path (D256 with at most 16 rows
    per sequence) and on the row path (D512, G 16)."""
    _, harness = kvq
    spec = _spec(8, 2, 256, 512, 256)
    wl = W.PrefillWorkload("verify-sliding", 84, spec, filled=[100, 700, 5, 1030], chunk=[2, 7, 33, 64],
                           bits=[4, 8, 8, 4])
    check_prefill(harness, wl)
    wl = W.PrefillWorkload("verify-sliding-rows", 84, spec, filled=[100, 700, 5, 1030, 511], chunk=[2, 7, 16, 1, 4],
                           bits=[4, 8, 8, 4, 8])
    check_prefill(harness, wl)
    spec = _spec(16, 1, 512, 0, 128, 1e6, True)
    wl = W.PrefillWorkload("verify-full", 85, spec, filled=[90, 3], chunk=[5, 17], bits=[8, 4])
    check_prefill(harness, wl)


def test_prefill_empty_sequences(kvq):
    """Sequences with no new rows inside a prompt call (first, middle and
    last), on the tensor-core path and on the row path, and a call with no
    rows at all: the other sequences' rows, caches and outputs are as the
    oracle has them."""
    _, harness = kvq
    wl = W.PrefillWorkload("empty-seqs-tc", 91, _spec(8, 2, 256, 64, 256), filled=[10, 100, 0, 7],
                           chunk=[0, 20, 0, 5], bits=[4, 8, 8, 4])
    check_prefill(harness, wl)
    wl = W.PrefillWorkload("empty-seqs-rows", 92, _spec(16, 1, 512, 0, 128, 1e6, True), filled=[30, 5, 64],
                           chunk=[3, 0, 0], bits=[8, 4, 8])
    check_prefill(harness, wl)
    wl = W.PrefillWorkload("no-rows", 93, _spec(8, 2, 256, 64, 256), filled=[10, 3], chunk=[0, 0], bits=[4, 8])
    check_prefill(harness, wl)


def test_prefill_row_path_gqa3(kvq):
    """A GQA ratio that does not divide the tensor-core kernel's 128 rows
    (G = 3) takes the row path for a prompt chunk on a window layer."""
    _, harness = kvq
    spec = W.LayerSpec(6, 2, 128, 48, 128, 1e4, False)
    wl = W.PrefillWorkload("gqa3-rows", 90, spec, filled=[30, 0], chunk=[20, 9], bits=[8, 4])
    check_prefill(harness, wl)


PREFILL_TC_CASES = {
    # name: (spec, filled per seq, chunk per seq, bits per seq) -- tensor-core path shapes
    "g1-d64": (_spec(2, 2, 64, 0, 64), [70, 3], [130, 9], [8, 4]),
    "g2-d128-window": (_spec(4, 2, 128, 96, 64, 1e6), [200, 0], [70, 45], [4, 8]),
    "g8-d256": (_spec(8, 1, 256, 0, 256), [31, 140], [40, 17], [8, 4]),
    "g16-d128-norope": (_spec(16, 1, 128, 0, 0), [64, 5], [24, 8], [4, 8]),
    "g16-d64-window": (_spec(32, 2, 64, 48, 64), [90, 3], [40, 11], [8, 4]),
    # the sliding-layer (dequantize-once) path at the other G and head_dim
    "g1-d64-window": (_spec(2, 2, 64, 40, 64), [70, 3], [130, 9], [8, 4]),
    "g8-d256-window": (_spec(8, 1, 256, 100, 256), [31, 140], [40, 17], [8, 4]),
    "g16-d128-window-norope": (_spec(16, 1, 128, 30, 0), [64, 5], [24, 8], [4, 8]),
}


@pytest.mark.parametrize("name", sorted(PREFILL_TC_CASES))
def test_prefill_tc_shapes(kvq, name):
    """The tensor-core prompt kernel across G (rows = 128/G tokens x G heads)
    and head_dim, full and windowed, with and without RoPE."""
    _, harness = kvq
    spec, filled, chunk, bits = PREFILL_TC_CASES[name]
    wl = W.PrefillWorkload(name, 86, spec, filled=filled, chunk=chunk, bits=bits)
    _, worst = check_prefill(harness, wl)
    print(name, "worst", worst)


def _bits32(t):
    """A tensor's bytes as int32 (NaN rows compare equal bit for bit)."""
    return t.contiguous().view(torch.int32) if t.element_size() == 4 else t.contiguous().view(torch.int16)


# attn_prefill_append: the chunk's append and read in one call, bit-equal to
# kv_quant_append + attn_prefill_chunk on each path: the dequantize-once
# tensor-core path (sliding), the codes-in-MMA tensor-core path (full, D128),
# the row path (D512; verify windows of at most 16 rows), and a chunk longer
# than its window ring (rows whose window reaches an overwritten key: NaN).
PREFILL_FUSED_CASES = {
    "sliding-prompt-tc": (_spec(8, 2, 256, 512, 256), [300, 0, 1000], [37, 130, 64], [8, 4, 4]),
    "full-d128-prefill-tc": (_spec(8, 1, 128, 0, 128, 1e6), [200, 5], [40, 17], [4, 8]),
    "full-keqv-d512-rows": (_spec(16, 1, 512, 0, 128, 1e6, True), [90, 3], [5, 17], [8, 4]),
    "verify-sliding-rows": (_spec(8, 2, 256, 512, 256), [100, 700, 0], [4, 16, 1], [4, 8, 8]),
}


@pytest.mark.parametrize("name", sorted(PREFILL_FUSED_CASES) + ["ring-overflow"])
def test_prefill_append_equals_separate_calls(kvq, name):
    _, harness = kvq
    if name == "ring-overflow":
        wl = W.PrefillWorkload("fused-overflow", 98, _spec(4, 1, 128, 64, 128), filled=[10], chunk=[300], bits=[4])
        wl.capacity = lambda s: 192
        wl.cached_positions = lambda s: np.arange(0, 10)
    else:
        spec, filled, chunk, bits = PREFILL_FUSED_CASES[name]
        wl = W.PrefillWorkload("fused-" + name, 98, spec, filled=filled, chunk=chunk, bits=bits)
    a = harness.PrefillCase(wl, keep_prepped=True)
    b = harness.PrefillCase(wl, keep_prepped=True)
    a.step()
    b.append_attend()
    torch.cuda.synchronize()
    assert a.status_word() == b.status_word()
    for x, y in ((a.out, b.out), (a.q_prepped, b.q_prepped), (a.kv_prepped, b.kv_prepped)):
        assert torch.equal(_bits32(x), _bits32(y))
    for s_ in range(wl.n_seqs):
        for key in a.caches.seqs[s_]:
            assert torch.equal(a.caches.seqs[s_][key], b.caches.seqs[s_][key]), (s_, key)
    if name != "ring-overflow":
        verify_prefill(b, wl)


def test_prefill_append_skips_a_bad_sequence(kvq):
    """attn_prefill_append on the dequantize-once tensor-core path with one
    sequence whose descriptor is invalid: its cache and its rows' scratch are
    not written, its output rows are NaN, the status word says so, and the
    other sequences' outputs are those of the same call without it."""
    _, harness = kvq
    spec, filled, chunk, bits = PREFILL_FUSED_CASES["sliding-prompt-tc"]
    wl = W.PrefillWorkload("fused-prefill-bad", 99, spec, filled=filled, chunk=chunk, bits=bits)
    c = harness.PrefillCase(wl)
    good = harness.PrefillCase(wl)
    torch.cuda.synchronize()
    before = c.caches.seqs[1]["k_codes"].clone()
    bad = c.caches.desc.cpu().numpy().copy()
    bad[56 + 48:56 + 52] = np.frombuffer(np.int32(5).tobytes(), np.uint8)      # seq 1: bits = 5
    c.caches.desc.copy_(torch.from_numpy(bad))
    c.append_attend()
    good.append_attend()
    torch.cuda.synchronize()
    assert c.status_word() & (1 << 2)
    assert torch.equal(before, c.caches.seqs[1]["k_codes"])
    r0, r1 = chunk[0], chunk[0] + chunk[1]
    out = c.out.cpu().numpy()
    assert np.all(np.isnan(out[r0:r1]))
    keep = list(range(r0)) + list(range(r1, sum(chunk)))
    assert torch.equal(_bits32(c.out[keep]), _bits32(good.out[keep]))


def test_prefill_bf16_output_is_rounded_f32(kvq):
    _, harness = kvq
    spec = _spec(8, 2, 256, 64, 256)
    wl = W.PrefillWorkload("prefill-bf16", 87, spec, filled=[150, 0], chunk=[100, 37], bits=[8, 4])
    a = harness.PrefillCase(wl)
    a.step()
    b = harness.PrefillCase(wl, out_f32=False)
    b.step()
    torch.cuda.synchronize()
    f32 = a.out.cpu().numpy()
    bf = b.out.cpu().numpy().view(np.uint16)
    want = O.f64_to_bf16(O.rn_bf16(f32.astype(np.float64)))
    assert np.array_equal(bf, want)


# ----------------------------------------------------------------------------
# mixed steps: decode groups and prompt / verify-window groups of one layer in
# one attn_mixed call, each group checked against the oracle on its own
# ----------------------------------------------------------------------------

# Each case: the layer, its groups, and the groups attn_mixed_schedule puts in
# the grouped decode-kernel launch (bit i = group i).
MIXED_CASES = {
    "sliding-decode-and-chunk": (_spec(8, 2, 256, 512, 256), [
        ("decode", [700, 40, 1500, 3], [4, 8, 8, 4]),
        ("window", [300, 0], [37, 130], [8, 4]),
    ], 0b00),
    "full-keqv-two-decode-one-verify": (_spec(16, 1, 512, 0, 128, 1e6, True), [
        ("decode", [3500, 10, 900], [8, 4, 4]),
        ("window", [200, 65], [5, 64], [4, 8]),
        ("decode", [64, 4000], [8, 8]),
    ], 0b111),
    # two decode groups and a verify window grouped; the prompt chunk on the
    # tensor cores beside them; an empty window group
    "sliding-grouped-decode-verify-beside-chunk": (_spec(8, 2, 256, 512, 256), [
        ("decode", [700, 40, 1500, 3, 511, 512], [4, 8, 8, 4, 8, 4]),
        ("window", [300, 5, 0], [4, 16, 1], [8, 4, 8]),
        ("window", [200, 0], [37, 130], [8, 4]),
        ("decode", [64, 900, 2000], [8, 4, 4]),
        ("window", [10], [0], [4]),
    ], 0b01011),
    # GQA 16 at head_dim 128, full causal: long ragged decode rows (the
    # standalone call would take stream-K) beside verify windows
    "d128-gqa16-grouped": (_spec(32, 2, 128, 0, 64, 1e6), [
        ("decode", [4000, 1, 64, 2500], [8, 4, 4, 8]),
        ("window", [3000, 63], [16, 2], [4, 8]),
    ], 0b11),
    # the deferred TurboQuant read: the grouped merge un-rotates every group
    "rot-full-keqv-grouped": (dataclasses.replace(_spec(16, 1, 512, 0, 128, 1e6, True), **ROT), [
        ("decode", [1200, 64, 3000], [4, 8, 4]),
        ("window", [100, 700], [3, 9], [8, 4]),
    ], 0b11),
}


@pytest.mark.parametrize("name", sorted(MIXED_CASES))
def test_mixed_groups(kvq, name):
    m, harness = kvq
    spec, groups, grouped = MIXED_CASES[name]
    wls = []
    for i, g in enumerate(groups):
        if g[0] == "decode":
            wls.append(W.DecodeWorkload(f"{name}-{i}", 91, spec, filled=g[1], bits=g[2]))
        else:
            wls.append(W.PrefillWorkload(f"{name}-{i}", 91, spec, filled=g[1], chunk=g[2], bits=g[3]))
    case = harness.MixedCase(wls, keep_prepped=True)
    assert m.attn_mixed_schedule(case.lay, case.groups(), case.q_w, case.out_f32) == grouped
    case.step()
    torch.cuda.synchronize()
    for c, wl in zip(case.cases, wls):
        if isinstance(wl, W.DecodeWorkload):
            worst = verify_decode(c, wl, check_fill=False)
        else:
            if c.n_rows:                # a group with no rows enqueues nothing
                assert c.status_word() == 0
            worst = verify_prefill(c, wl)
        print(name, wl.name, "worst", worst)


def test_mixed_equals_separate_calls(kvq):
    """Groups of an attn_mixed call that run on their own kernels (here a
    decode group beside a prompt chunk on the tensor cores: nothing to group)
    give the same bytes as the separate attn_decode / attn_prefill_chunk
    calls."""
    m, harness = kvq
    spec = _spec(8, 2, 256, 512, 256)
    wls = [W.DecodeWorkload("eq-d", 92, spec, filled=[900, 33], bits=[4, 8]),
           W.PrefillWorkload("eq-w", 92, spec, filled=[128], chunk=[70], bits=[8])]
    case = harness.MixedCase(wls)
    assert m.attn_mixed_schedule(case.lay, case.groups(), case.q_w, case.out_f32) == 0
    case.append()
    case.attend()
    torch.cuda.synchronize()
    mixed = [c.out.clone() for c in case.cases]
    case.attend_serial()
    torch.cuda.synchronize()
    for a, c in zip(mixed, case.cases):
        assert torch.equal(a, c.out)
