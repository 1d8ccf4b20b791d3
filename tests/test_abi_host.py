"""Host-side checks of the C ABI: the library loads, exports every function
include/kvq.h declares, and rejects bad arguments with the documented status
before enqueueing any GPU work (no compute call is made here)."""
import ctypes
import os
import shutil
import subprocess

import pytest


@pytest.fixture(scope="module")
def m():
    import __graft_entry__
    __graft_entry__.build()
    import quantized_kv_attention_quant_gb300 as pkg
    return pkg


def test_exports_every_declared_function(m):
    names = m.header_functions()
    assert set(names) >= {"kv_quant_append", "attn_decode", "attn_prefill_chunk",
                          "attn_decode_workspace_bytes", "attn_prefill_workspace_bytes",
                          "kvq_status_string", "kvq_last_error", "kvq_version"}
    lib = ctypes.CDLL(m.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"libkvq.so does not export {n}"


def test_status_strings_and_version(m):
    assert m.kvq_status_string(0) == "ok"
    for st in range(1, 5):
        assert m.kvq_status_string(st) not in ("ok", "unknown status")
    assert m.kvq_status_string(99) == "unknown status"
    assert m.kvq_version() >= 100


def test_struct_layout_matches_header(m):
    assert ctypes.sizeof(m.KvqSeqCache) == 56
    assert m.KvqSeqCache.bits.offset == 48 and m.KvqSeqCache.capacity.offset == 52
    assert m.KvqLayer.rope_theta.offset == 24 and m.KvqLayer.rot_signs.offset == 40
    assert ctypes.sizeof(m.KvqLayer) == 48


GOOD = dict(n_q_heads=8, n_kv_heads=2, head_dim=256, window=512, rope_dims=256, rope_theta=1e4)
P = 1 << 20          # a fake, aligned "device address": never dereferenced (calls fail on the host)


def _layer(m, **kw):
    d = dict(GOOD)
    d.update(kw)
    return m.layer(**d)


@pytest.mark.parametrize("kw,status", [
    (dict(n_q_heads=6, n_kv_heads=4), 1),       # not a multiple
    (dict(n_q_heads=0), 1),
    (dict(n_q_heads=34, n_kv_heads=2), 2),      # ratio 17 > 16
    (dict(head_dim=96), 2),
    (dict(head_dim=1024), 2),
    (dict(window=-1), 1),
    (dict(rope_dims=3), 1),
    (dict(rope_dims=512), 1),
    (dict(rope_theta=0.0), 1),
    (dict(rope_theta=float("inf")), 1),
])
def test_bad_layer(m, kw, status):
    lay = _layer(m, **kw)
    st = m.lib.kv_quant_append(ctypes.byref(lay), P, 1, P, P, 1, P, P, P, None, None)
    assert st == status
    assert m.kvq_last_error()
    assert m.attn_decode_workspace_bytes(lay, 1, 10) == 0


def test_bad_group_and_eps(m):
    lay = _layer(m)
    lay.group_size = 32
    assert m.lib.attn_decode(ctypes.byref(lay), P, 1, P, 10, P, P, P, 1, None, P, 1 << 30, None) == 2
    lay = _layer(m, rms_eps=-1.0)
    assert m.lib.attn_decode(ctypes.byref(lay), P, 1, P, 10, P, P, P, 1, None, P, 1 << 30, None) == 1
    assert m.lib.attn_decode(None, P, 1, P, 10, P, P, P, 1, None, P, 1 << 30, None) == 1


def test_bad_pointers_append(m):
    lay = _layer(m)
    f = m.lib.kv_quant_append
    L = ctypes.byref(lay)
    assert f(L, None, 1, P, P, 1, P, P, P, None, None) == 1            # seqs NULL
    assert f(L, P + 4, 1, P, P, 1, P, P, P, None, None) == 1           # seqs misaligned
    assert f(L, P, 1, P, P, 1, P + 8, P, P, None, None) == 1           # k_raw not 16-aligned
    assert f(L, P, 1, P, P, 1, P, None, P, None, None) == 1            # v_raw missing
    keqv = _layer(m, k_eq_v=True)
    assert f(ctypes.byref(keqv), P, 1, P, P, 1, P, P, P, None, None) == 1   # v_raw given with K = V
    assert f(L, P, 1, P, P, 1, P, P, P, P + 1, None) == 1              # kv_prepped odd address
    assert f(L, P, -1, P, P, 1, P, P, P, None, None) == 1
    assert f(L, P, 0, P, P, 1, P, P, P, None, None) == 1               # rows without sequences
    assert f(L, P, 1, P, P, 0, P, P, P, None, None) == 0               # nothing to do


def test_bad_pointers_decode(m):
    lay = _layer(m)
    f = m.lib.attn_decode
    L = ctypes.byref(lay)
    big = 1 << 40
    assert f(L, P, 1, P, 10, P + 8, P, P, 1, None, P, big, None) == 1     # q_raw misaligned
    assert f(L, P, 1, None, 10, P, P, P, 1, None, P, big, None) == 1      # pos NULL
    assert f(L, P, 1, P, 10, P, P, P + 2, 1, None, P, big, None) == 1     # f32 out misaligned
    assert f(L, P, 1, P, 10, P, P, P, 2, None, P, big, None) == 1         # out_is_f32 not 0/1
    assert f(L, P, 1, P, 10, P, P, P, 1, None, P + 16, big, None) == 1    # workspace not 256-aligned
    assert f(L, P, 1, P, -1, P, P, P, 1, None, P, big, None) == 1         # max_pos < 0
    assert f(L, P, 1, P, 1 << 24, P, P, P, 1, None, P, big, None) == 1    # max_pos >= 2^24
    assert f(L, P, 1, P, 2 ** 31 - 1, P, P, P, 1, None, P, big, None) == 1
    assert m.attn_decode_workspace_bytes(lay, 1, 1 << 24) == 0
    assert m.attn_decode_workspace_bytes(lay, 1, 2 ** 31 - 1) == 0
    assert m.attn_decode_workspace_bytes(lay, 1, (1 << 24) - 1) > 0
    assert m.lib.attn_decode_static(L, P, 1, P, 2 ** 31 - 1, P, P, P, 1, None, None) == 1
    need = m.attn_decode_workspace_bytes(lay, 1, 10)
    assert need > 0
    assert f(L, P, 1, P, 10, P, P, P, 1, None, P, need - 1, None) == 4    # workspace too small
    assert f(L, P, 0, P, 10, P, P, P, 1, None, P, 0, None) == 0           # no sequences: no work


def test_bad_pointers_decode_append(m):
    """attn_decode_append checks the decode half and the append half before
    enqueueing anything."""
    lay = _layer(m)
    f = m.lib.attn_decode_append
    L = ctypes.byref(lay)
    big = 1 << 40
    # (layer, seqs, n, pos, max_pos, q, k, v, q_w, k_w, out, f32, q_prepped, kv_prepped, ws, ws_bytes, stream)
    assert f(L, P, 1, P, -1, P, P, P, P, P, P, 1, None, None, P, big, None) == 1     # max_pos < 0
    assert f(L, P, 1, P, 10, P + 8, P, P, P, P, P, 1, None, None, P, big, None) == 1  # q_raw misaligned
    assert f(L, P, 1, P, 10, P, None, P, P, P, P, 1, None, None, P, big, None) == 1   # k_raw NULL
    assert f(L, P, 1, P, 10, P, P + 8, P, P, P, P, 1, None, None, P, big, None) == 1  # k_raw misaligned
    assert f(L, P, 1, P, 10, P, P, None, P, P, P, 1, None, None, P, big, None) == 1   # v_raw missing
    assert f(L, P, 1, P, 10, P, P, P, P, None, P, 1, None, None, P, big, None) == 1   # k_norm_w NULL
    assert f(L, P, 1, P, 10, P, P, P, P, P, P, 1, None, P + 1, P, big, None) == 1     # kv_prepped odd
    keqv = _layer(m, k_eq_v=True)
    assert f(ctypes.byref(keqv), P, 1, P, 10, P, P, P, P, P, P, 1, None, None, P, big, None) == 1  # v_raw with K=V
    need = m.attn_decode_workspace_bytes(lay, 1, 10)
    assert f(L, P, 1, P, 10, P, P, P, P, P, P, 1, None, None, P, need - 1, None) == 4  # workspace too small
    assert f(L, P, 0, P, 10, P, P, P, P, P, P, 1, None, None, P, 0, None) == 0        # no sequences


def test_bad_pointers_prefill(m):
    lay = _layer(m)
    f = m.lib.attn_prefill_chunk
    L = ctypes.byref(lay)
    assert f(L, P, 1, None, P, 4, 4, P, P, P, 1, None, P, 1 << 40, None) == 1   # row_offsets NULL
    assert f(L, P, 1, P, P, 4, 0, P, P, P, 1, None, P, 1 << 40, None) == 1      # max_rows < 1
    need = m.attn_prefill_workspace_bytes(lay, 1, 4, 4)
    assert need > 0
    assert f(L, P, 1, P, P, 4, 4, P, P, P, 1, None, P, need - 1, None) == 4


def test_workspace_grows_with_rows(m):
    lay = _layer(m)
    assert m.attn_prefill_workspace_bytes(lay, 1, 64, 64) < m.attn_prefill_workspace_bytes(lay, 1, 512, 512)
    full = _layer(m, window=0, head_dim=512, n_q_heads=16, n_kv_heads=1, rope_dims=128)
    assert m.attn_decode_workspace_bytes(full, 8, 32768) > 0


def test_bad_mixed_groups(m):
    """attn_mixed checks every group before enqueueing anything."""
    lay = _layer(m)
    L = ctypes.byref(lay)
    big = 1 << 40
    dec = m.attn_group(m.KVQ_PHASE_DECODE, P, 1, None, P, 0, 10, 0, P, P, None, P, big)
    win = m.attn_group(m.KVQ_PHASE_WINDOW, P, 1, P, P, 4, 0, 4, P, P, None, P + (1 << 30), big)
    f = m.lib.attn_mixed

    def call(groups, n=None):
        arr = (m.KvqAttnGroup * max(1, len(groups)))(*groups)
        return f(L, arr, len(groups) if n is None else n, P, 1, None)

    assert call([], 0) == 0                                       # nothing to do
    assert call([dec] * 9) == 1                                   # more than KVQ_MAX_MIXED_GROUPS
    assert f(L, None, 1, P, 1, None) == 1                         # groups NULL
    bad_phase = m.attn_group(7, P, 1, None, P, 0, 10, 0, P, P, None, P, big)
    assert call([dec, bad_phase]) == 1
    assert "group 1" in m.kvq_last_error()
    bad_pos = m.attn_group(m.KVQ_PHASE_DECODE, P, 1, None, P, 0, -1, 0, P, P, None, P, big)
    assert call([bad_pos]) == 1
    far_pos = m.attn_group(m.KVQ_PHASE_DECODE, P, 1, None, P, 0, 2 ** 31 - 1, 0, P, P, None, P, big)
    assert call([win, far_pos]) == 1 and "group 1" in m.kvq_last_error()
    no_offsets = m.attn_group(m.KVQ_PHASE_WINDOW, P, 1, None, P, 4, 0, 4, P, P, None, P, big)
    assert call([dec, no_offsets]) == 1
    misaligned = m.attn_group(m.KVQ_PHASE_DECODE, P, 1, None, P, 0, 10, 0, P + 8, P, None, P, big)
    assert call([win, misaligned]) == 1                           # q_raw of group 1 misaligned
    small = m.attn_group(m.KVQ_PHASE_WINDOW, P, 1, P, P, 4, 0, 4, P, P, None, P,
                         m.attn_prefill_workspace_bytes(lay, 1, 4, 4) - 1)
    assert call([dec, small]) == 4                                # workspace too small
    assert call([dec, dec]) == 1                                  # the same workspace twice
    assert "share workspace" in m.kvq_last_error()


def test_mixed_grouped_schedule_membership(m):
    """attn_mixed_schedule: decode groups, verify windows (at most 16 rows
    per sequence, read by the decode kernels) and window groups no
    tensor-core kernel takes share the grouped launch; larger prompt chunks on
    the tensor cores, empty groups and groups whose workspace holds no split
    of the shared plan run on their own."""
    big = 1 << 36

    def grp(k, phase, n_seqs, n_rows=0, max_pos=0, max_rows=0, ws=big):
        base = P + k * (1 << 40)                  # disjoint workspaces
        return m.attn_group(phase, P, n_seqs, P if phase == m.KVQ_PHASE_WINDOW else None, P, n_rows, max_pos,
                            max_rows, P, P, None, base, ws)

    def mask(lay, groups):
        return m.attn_mixed_schedule(lay, groups, P, 1)

    D, W_ = m.KVQ_PHASE_DECODE, m.KVQ_PHASE_WINDOW
    sliding = _layer(m)                           # 8q/2kv D256 W512: prompt chunks on the tensor cores
    assert mask(sliding, []) == 0
    assert mask(sliding, [grp(0, D, 48, max_pos=8000)]) == 0
    assert mask(sliding, [grp(0, D, 48, max_pos=8000), grp(1, D, 3, max_pos=10)]) == 0b11
    verify, chunk = grp(1, W_, 8, 32, max_rows=4), grp(2, W_, 2, 512, max_rows=256)
    assert mask(sliding, [grp(0, D, 48, max_pos=8000), verify, chunk]) == 0b011
    assert mask(sliding, [grp(0, D, 48, max_pos=8000), chunk]) == 0      # one member: nothing to group
    assert mask(sliding, [verify, grp(3, W_, 4, 64, max_rows=16), chunk]) == 0b011
    assert mask(sliding, [verify, grp(3, W_, 4, 68, max_rows=17)]) == 0  # 17 rows: the tensor cores
    empty = grp(3, W_, 1, 0, max_rows=0)
    assert mask(sliding, [grp(0, D, 48, max_pos=8000), empty, verify]) == 0b101
    full = _layer(m, window=0, head_dim=512, n_q_heads=16, n_kv_heads=1, rope_dims=128)
    # head_dim 512: every window group is read by the decode kernels
    assert mask(full, [grp(0, D, 8, max_pos=32767), grp(1, W_, 2, 512, max_rows=256)]) == 0b11
    # a decode group sized for its own stream-K plan: 512 rows need 512 pieces
    # even at one split, its workspace holds 2 per stream-K CTA
    own = m.attn_decode_workspace_bytes(full, 512, 32767)
    wide = grp(0, D, 512, max_pos=32767, ws=own)
    assert mask(full, [wide, grp(1, D, 8, max_pos=100), grp(2, D, 4, max_pos=50)]) == 0b110
    assert mask(full, [wide, grp(1, D, 8, max_pos=100)]) == 0
    assert mask(full, [grp(0, D, 512, max_pos=32767), grp(1, D, 8, max_pos=100)]) == 0b11
    # a verify window sized by attn_prefill_workspace_bytes joins (head_dim
    # 128, GQA 16, full causal)
    d128 = _layer(m, window=0, head_dim=128, n_q_heads=32, n_kv_heads=2, rope_dims=64)
    vws = m.attn_prefill_workspace_bytes(d128, 2, 18, 16)
    assert mask(d128, [grp(0, D, 4, max_pos=4000), grp(1, W_, 2, 18, max_rows=16, ws=vws)]) == 0b11
    assert mask(d128, [grp(0, D, 4, max_pos=4000), grp(1, W_, 2, 34, max_rows=17)]) == 0
    # the checks of attn_mixed come first
    with pytest.raises(RuntimeError):
        mask(sliding, [grp(0, D, 48, max_pos=8000), grp(0, D, 3, max_pos=10)])   # shared workspace
    assert m.lib.attn_mixed_schedule(ctypes.byref(sliding), None, 0, P, 1, None) == 1


def test_prompt_workspace_holds_the_dequantized_window(m):
    """Sliding layers' prompt calls (more than 16 rows per sequence) keep
    k_hi, k_lo and v (f16) of window + rows - 1 keys per sequence (whole
    64-key tiles) besides q_hat as f16; full layers' prompt calls keep no such
    scratch."""
    lay = _layer(m)                                   # 8q/2kv, D256, window 512
    def expect(n_seqs, n_rows, max_rows, window=512, hkv=2, hq=8, d=256):
        ks = -(-(window + max_rows - 1) // 64) * 64
        scratch = n_seqs * ks * hkv * d * 2
        a256 = lambda x: (x + 255) & ~255
        off = a256(256 + n_rows * hq * d * 2)
        off = a256(off + scratch)
        off = a256(off + scratch)
        return off + scratch
    for n_seqs, n_rows, max_rows in ((1, 17, 17), (4, 2048, 512), (3, 100, 64)):
        assert m.attn_prefill_workspace_bytes(lay, n_seqs, n_rows, max_rows) == expect(n_seqs, n_rows, max_rows)
    # verify windows (at most 16 rows per sequence) take the decode kernels'
    # workspace (q fragments and split partials), not the dequantized window
    assert m.attn_prefill_workspace_bytes(lay, 1, 16, 16) not in (0, expect(1, 16, 16))
    full = _layer(m, window=0)
    assert m.attn_prefill_workspace_bytes(full, 4, 2048, 512) < expect(4, 2048, 512)


def test_bad_selftest_arguments(m):
    f = m.lib.kvq_selftest_wait_timeout
    assert f(None, 1000000, None) == 1            # status NULL
    assert f(P + 2, 1000000, None) == 1           # status misaligned
    assert f(P, 10, None) == 1                    # limit below 1 us
    assert f(P, 2000000000, None) == 1            # limit above 1 s
    g = m.lib.kvq_static_status
    assert g(None, None) == 1                     # status NULL
    assert g(P + 2, None) == 1                    # status misaligned


def test_bad_training_arguments(m):
    lay = _layer(m)
    L = ctypes.byref(lay)
    f = m.lib.attn_train_forward
    need = m.attn_train_workspace_bytes(lay, 100)
    assert need == 256 + 100 * 8 * 256 * 2
    big = 1 << 40
    ok = (L, 2, P, 100, 60, P, P, P, P, P, 1, None, P, big, None)

    def call(**kw):
        a = list(ok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return f(*a)
    assert call(a1=0) == 1                                    # no block
    assert call(a1=65536) == 1
    assert call(a2=None) == 1                                 # block_offsets NULL
    assert call(a3=1 << 24) == 1                              # rows past the position range
    assert call(a4=0) == 1 and call(a4=101) == 1              # max_block_rows out of [1, n_rows]
    assert call(a5=P + 8) == 1                                # q_raw not 16-aligned
    assert call(a7=P + 2) == 1 and call(a8=P + 2) == 1        # k_hat, v_hat not 16-aligned
    assert call(a9=P + 2) == 1                                # f32 out misaligned
    assert call(a10=2) == 1                                   # out_is_f32 not 0/1
    assert call(a12=P + 16) == 1                              # workspace not 256-aligned
    assert call(a13=need - 1) == 4                            # workspace too small
    rot = _layer(m, rot_signs=P)
    assert f(ctypes.byref(rot), *ok[1:]) == 2                 # no rotated training read
    g3 = _layer(m, n_q_heads=6, n_kv_heads=2)
    assert f(ctypes.byref(g3), *ok[1:]) == 2                  # 3 q heads per kv head do not divide 128
    assert call(a3=0) == 0                                    # no rows: nothing to do
    p = m.lib.kvq_train_kv_prep
    assert p(L, 2, P, 100, P, P, P, P + 2, P, None) == 1      # k_hat misaligned
    assert p(L, 2, P, 100, P, None, P, P, P, None) == 1       # v_raw missing
    keqv = _layer(m, k_eq_v=True)
    assert p(ctypes.byref(keqv), 2, P, 100, P, P, P, P, P, None) == 1   # v_raw given with K = V
    assert p(ctypes.byref(rot), 2, P, 100, P, P, P, P, P, None) == 2
    assert p(L, 2, None, 100, P, P, P, P, P, None) == 1
    assert p(L, 2, P, 0, P, P, P, P, P, None) == 0


def test_plain_c_program(m, tmp_path):
    """include/kvq.h compiles as pedantic C11 and a C program links libkvq.so,
    resolves every declared function and gets the documented host-side
    results (tests/c_abi_check.c)."""
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    here = os.path.dirname(os.path.abspath(__file__))
    root = os.path.dirname(here)
    libdir = os.path.dirname(m.LIB_PATH)
    exe = str(tmp_path / "c_abi_check")
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I" + os.path.join(root, "include"), os.path.join(here, "c_abi_check.c"),
                    "-L" + libdir, "-lkvq", "-Wl,-rpath," + libdir, "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout[-2000:]
    assert r.stdout.strip().endswith("all checks passed")
