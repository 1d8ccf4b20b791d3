"""A sequence's life through consecutive calls on the GPU, against the float64
oracle stepping the same way: a prompt chunk, a verify window, then decode
steps whose ring wraps, on a sliding layer (4- and 8-bit caches side by side)
and on a full K = V layer.  Every call's prepped rows bit-exact, every
output within max-abs 1e-2 / mean-abs 1e-3, the cache bytes bit-exact at the
end.  The calls carry state only in the caches, so a mistake in a ring slot,
a position or a partially written tile shows up in a later call."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from oracle_ref import attn_errors, compare_cache, oracle_layer, ring_slots

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 1e-2, 1e-3
P_STEP = 40           # a stream purpose of its own for these inputs


@pytest.fixture(scope="module")
def kvq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_kv_attention_quant_gb300 as m
    from quantized_kv_attention_quant_gb300 import harness
    return m, harness


def _bits(t):
    return t.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("kind", ["sliding", "full"])
def test_prompt_verify_then_decode(kvq, kind):
    m, harness = kvq
    if kind == "sliding":
        spec = W.LayerSpec(8, 2, 256, 96, 256, 1e4, False)
        prompt, caps = [150, 70], [192, 192]          # rings of window + rows - 1 or more
    else:
        spec = W.LayerSpec(16, 1, 512, 0, 128, 1e6, True)
        prompt, caps = [130, 9], [320, 320]
    bits = [4, 8]
    verify, steps = [5, 12], 40                       # the sliding rings wrap during the decode steps
    n = 2
    seed = 1301
    dev = "cuda"
    L = oracle_layer(spec)
    lay = harness.kvq_layer(spec)
    Hq, Hkv, D = spec.n_q_heads, spec.n_kv_heads, spec.head_dim
    caches = harness.LayerCaches(Hkv, D, bits, caps, dev)
    w = W.layer_inputs(seed, 0, spec, 0, 0)
    q_w, k_w = harness.dev_bits(w["q_w"], dev), harness.dev_bits(w["k_w"], dev)
    f = O.bf16_to_f64
    ocache = [O.OracleCache(Hkv, D, b) for b in bits]
    pos = [0, 0]

    def draws(call, rows):
        q = W.normal_bf16(seed, (P_STEP, call, 0), (rows, Hq, D))
        k = W.normal_bf16(seed, (P_STEP, call, 1), (rows, Hkv, D))
        v = None if spec.k_eq_v else W.normal_bf16(seed, (P_STEP, call, 2), (rows, Hkv, D))
        return q, k, v

    def window_call(call, chunk):
        rows = int(sum(chunk))
        q, k, v = draws(call, rows)
        offs = harness.dev_i32(np.concatenate([[0], np.cumsum(chunk)]), dev)
        start = harness.dev_i32(pos, dev)
        kvp = torch.empty((2, rows, Hkv, D), dtype=torch.int16, device=dev)
        qp = torch.empty((rows, Hq, D), dtype=torch.int16, device=dev)
        out = torch.empty((rows, Hq, D), dtype=torch.float32, device=dev)
        wsb = m.attn_prefill_workspace_bytes(lay, n, rows, max(chunk))
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        qd, kd = harness.dev_bits(q, dev), harness.dev_bits(k, dev)
        vd = harness.dev_bits(v, dev) if v is not None else None
        m.kv_quant_append(lay, caches.desc, n, offs, start, rows, kd, vd, k_w, kvp)
        m.attn_prefill_chunk(lay, caches.desc, n, offs, start, rows, max(chunk), qd, q_w, out, 1, qp, ws, wsb)
        torch.cuda.synchronize()
        assert int(ws[:4].cpu().numpy().view(np.uint32)[0]) == 0
        o, qpb, kvb = out.cpu().numpy(), _bits(qp), _bits(kvp)
        r0 = 0
        for s in range(n):
            sl = slice(r0, r0 + chunk[s])
            q_hat, k_hat, v_hat, outs = O.prefill_chunk(L, ocache[s], pos[s], f(q[sl]), f(w["q_w"]), f(k[sl]),
                                                        None if v is None else f(v[sl]), f(w["k_w"]))
            assert np.array_equal(qpb[sl], O.f64_to_bf16(q_hat)), (call, s, "q prep")
            assert np.array_equal(kvb[0, sl], O.f64_to_bf16(k_hat)) and np.array_equal(kvb[1, sl], O.f64_to_bf16(v_hat))
            for t, want in outs.items():
                mx, mean = attn_errors(o[r0 + t], want)
                assert mx <= MAX_ABS and mean <= MEAN_ABS, (call, s, t, mx, mean)
            r0 += chunk[s]
            pos[s] += chunk[s]

    def decode_call(call):
        q, k, v = draws(call, n)
        p = harness.dev_i32(pos, dev)
        offs = harness.dev_i32(np.arange(n + 1), dev)
        kvp = torch.empty((2, n, Hkv, D), dtype=torch.int16, device=dev)
        qp = torch.empty((n, Hq, D), dtype=torch.int16, device=dev)
        out = torch.empty((n, Hq, D), dtype=torch.float32, device=dev)
        wsb = m.attn_decode_workspace_bytes(lay, n, max(pos))
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        qd, kd = harness.dev_bits(q, dev), harness.dev_bits(k, dev)
        vd = harness.dev_bits(v, dev) if v is not None else None
        m.kv_quant_append(lay, caches.desc, n, offs, p, n, kd, vd, k_w, kvp)
        m.attn_decode(lay, caches.desc, n, p, max(pos), qd, q_w, out, 1, qp, ws, wsb)
        torch.cuda.synchronize()
        assert int(ws[:4].cpu().numpy().view(np.uint32)[0]) == 0
        o, qpb, kvb = out.cpu().numpy(), _bits(qp), _bits(kvp)
        for s in range(n):
            q_hat, k_hat, v_hat, want = O.decode_step(L, ocache[s], pos[s], f(q[s]), f(w["q_w"]), f(k[s]),
                                                      None if v is None else f(v[s]), f(w["k_w"]))
            assert np.array_equal(qpb[s], O.f64_to_bf16(q_hat)), (call, s, "q prep")
            assert np.array_equal(kvb[0, s], O.f64_to_bf16(k_hat)) and np.array_equal(kvb[1, s], O.f64_to_bf16(v_hat))
            mx, mean = attn_errors(o[s], want)
            assert mx <= MAX_ABS and mean <= MEAN_ABS, (call, s, mx, mean)
            pos[s] += 1

    window_call(0, prompt)
    window_call(1, verify)
    for i in range(steps):
        decode_call(2 + i)
    for s in range(n):
        newest = pos[s] - 1
        resident = np.arange(max(0, newest - caps[s] + 1), newest + 1)
        rows = caches.host_rows(s, ring_slots(resident, caps[s]))
        assert compare_cache(rows, ocache[s], resident) == 0, f"seq {s}: cache bytes"
