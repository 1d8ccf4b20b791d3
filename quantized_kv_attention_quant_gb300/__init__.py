"""Python binding of libkvq.so: attention over a group-wise affine-quantized
KV cache on one GB300 GPU (sm_103a).

The functions below carry the C ABI's names (include/kvq.h) and only marshal
arguments: every step of the computation runs in the library's CUDA kernels.
Tensor arguments may be torch tensors (their data pointers are passed) or raw
integer device addresses.  A failing call raises KvqError.  Importing this
package without a built library raises ImportError: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkvq.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "kvq.h")

KVQ_OK, KVQ_EINVAL, KVQ_EUNSUPPORTED, KVQ_ECUDA, KVQ_EWORKSPACE = range(5)
# bits of the device status word left in the first 4 bytes of a workspace
KVQ_STATUS_WAIT_TIMEOUT, KVQ_STATUS_SEQ_SKIPPED = 0x2, 0x4


class KvqLayer(ctypes.Structure):
    _fields_ = [("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("group_size", ctypes.c_int32),
                ("window", ctypes.c_int32), ("rope_dims", ctypes.c_int32),
                ("rope_theta", ctypes.c_double), ("rms_eps", ctypes.c_float),
                ("k_eq_v", ctypes.c_int32), ("rot_signs", ctypes.c_void_p)]


class KvqSeqCache(ctypes.Structure):
    _fields_ = [("k_codes", ctypes.c_void_p), ("v_codes", ctypes.c_void_p),
                ("k_scales", ctypes.c_void_p), ("k_biases", ctypes.c_void_p),
                ("v_scales", ctypes.c_void_p), ("v_biases", ctypes.c_void_p),
                ("bits", ctypes.c_int32), ("capacity", ctypes.c_int32)]


KVQ_MAX_MIXED_GROUPS = 8
KVQ_PHASE_DECODE, KVQ_PHASE_WINDOW = 0, 1


class KvqAttnGroup(ctypes.Structure):
    _fields_ = [("phase", ctypes.c_int32), ("seqs", ctypes.c_void_p), ("n_seqs", ctypes.c_int32),
                ("row_offsets", ctypes.c_void_p), ("pos", ctypes.c_void_p), ("n_rows", ctypes.c_int32),
                ("max_pos", ctypes.c_int32), ("max_rows_per_seq", ctypes.c_int32),
                ("q_raw", ctypes.c_void_p), ("out", ctypes.c_void_p), ("q_prepped", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t)]


class KvqError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"kvq status {status}: {message}")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run "
                          "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    lay = ctypes.POINTER(KvqLayer)
    lib.kv_quant_append.argtypes = [lay, vp, i32, vp, vp, i32, vp, vp, vp, vp, vp]
    lib.kv_quant_append.restype = ctypes.c_int
    lib.attn_decode.argtypes = [lay, vp, i32, vp, i32, vp, vp, vp, i32, vp, vp, sz, vp]
    lib.attn_decode.restype = ctypes.c_int
    lib.attn_decode_append.argtypes = [lay, vp, i32, vp, i32, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, sz, vp]
    lib.attn_decode_append.restype = ctypes.c_int
    lib.attn_decode_static.argtypes = [lay, vp, i32, vp, i32, vp, vp, vp, i32, vp, vp]
    lib.attn_decode_static.restype = ctypes.c_int
    lib.attn_decode_workspace_bytes.argtypes = [lay, i32, i32]
    lib.attn_decode_workspace_bytes.restype = sz
    lib.attn_prefill_chunk.argtypes = [lay, vp, i32, vp, vp, i32, i32, vp, vp, vp, i32, vp, vp, sz, vp]
    lib.attn_prefill_chunk.restype = ctypes.c_int
    lib.attn_prefill_workspace_bytes.argtypes = [lay, i32, i32, i32]
    lib.attn_prefill_workspace_bytes.restype = sz
    lib.attn_mixed.argtypes = [lay, ctypes.POINTER(KvqAttnGroup), i32, vp, i32, vp]
    lib.attn_mixed.restype = ctypes.c_int
    lib.attn_mixed_schedule.argtypes = [lay, ctypes.POINTER(KvqAttnGroup), i32, vp, i32, vp]
    lib.attn_mixed_schedule.restype = ctypes.c_int
    lib.kvq_train_kv_prep.argtypes = [lay, i32, vp, i32, vp, vp, vp, vp, vp, vp]
    lib.kvq_train_kv_prep.restype = ctypes.c_int
    lib.attn_train_forward.argtypes = [lay, i32, vp, i32, i32, vp, vp, vp, vp, vp, i32, vp, vp, sz, vp]
    lib.attn_train_forward.restype = ctypes.c_int
    lib.attn_prefill_append.argtypes = [lay, vp, i32, vp, vp, i32, i32, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp,
                                        sz, vp]
    lib.attn_prefill_append.restype = ctypes.c_int
    lib.attn_train_donor_forward.argtypes = [lay, i32, vp, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp,
                                             sz, vp]
    lib.attn_train_donor_forward.restype = ctypes.c_int
    lib.attn_train_workspace_bytes.argtypes = [lay, i32]
    lib.attn_train_workspace_bytes.restype = sz
    lib.kvq_static_status.argtypes = [vp, vp]
    lib.kvq_static_status.restype = ctypes.c_int
    lib.kvq_selftest_wait_timeout.argtypes = [vp, ctypes.c_uint64, vp]
    lib.kvq_selftest_wait_timeout.restype = ctypes.c_int
    lib.kvq_profile_next_read.argtypes = [vp, vp]
    lib.kvq_profile_next_read.restype = ctypes.c_int
    lib.kvq_status_string.argtypes = [ctypes.c_int]
    lib.kvq_status_string.restype = ctypes.c_char_p
    lib.kvq_last_error.argtypes = []
    lib.kvq_last_error.restype = ctypes.c_char_p
    lib.kvq_version.argtypes = []
    lib.kvq_version.restype = i32
    return lib


lib = _load()


def header_functions() -> list:
    """Names of the functions include/kvq.h declares."""
    text = open(HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = "\n".join(ln for ln in text.splitlines() if not ln.lstrip().startswith("#"))
    return sorted(set(re.findall(r"\b([A-Za-z_]\w*)\s*\([^;{]*\)\s*;", text)) - {"if", "while"})


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, ctypes.Array):
        return ctypes.addressof(x)
    raise TypeError(f"cannot pass {type(x)} as a device pointer")


def _stream(stream):
    if stream is None:
        try:
            import torch
            if torch.cuda.is_available():
                return torch.cuda.current_stream().cuda_stream
        except ImportError:
            pass
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int):
    if status != KVQ_OK:
        raise KvqError(status, lib.kvq_last_error().decode())


def layer(n_q_heads, n_kv_heads, head_dim, window, rope_dims, rope_theta, rms_eps=1e-6,
          k_eq_v=False, group_size=64, rot_signs=None) -> KvqLayer:
    """rot_signs: None, or the device int8 [head_dim] signs of the deferred
    TurboQuant read (a tensor or an address; see include/kvq.h)."""
    return KvqLayer(n_q_heads, n_kv_heads, head_dim, group_size, window, rope_dims,
                    float(rope_theta), float(rms_eps), int(bool(k_eq_v)), _ptr(rot_signs))


def kv_quant_append(layer: KvqLayer, seqs, n_seqs, row_offsets, start_pos, n_rows, k_raw, v_raw,
                    k_norm_w, kv_prepped=None, stream=None):
    _check(lib.kv_quant_append(ctypes.byref(layer), _ptr(seqs), n_seqs, _ptr(row_offsets),
                               _ptr(start_pos), n_rows, _ptr(k_raw), _ptr(v_raw), _ptr(k_norm_w),
                               _ptr(kv_prepped), _stream(stream)))


def attn_decode(layer: KvqLayer, seqs, n_seqs, pos, max_pos, q_raw, q_norm_w, out, out_is_f32,
                q_prepped, workspace, workspace_bytes, stream=None):
    _check(lib.attn_decode(ctypes.byref(layer), _ptr(seqs), n_seqs, _ptr(pos), max_pos, _ptr(q_raw),
                           _ptr(q_norm_w), _ptr(out), int(out_is_f32), _ptr(q_prepped),
                           _ptr(workspace), workspace_bytes, _stream(stream)))


def attn_decode_append(layer: KvqLayer, seqs, n_seqs, pos, max_pos, q_raw, k_raw, v_raw, q_norm_w, k_norm_w,
                       out, out_is_f32, q_prepped, kv_prepped, workspace, workspace_bytes, stream=None):
    """kv_quant_append of one row per sequence at pos, then attn_decode, in one
    call (see include/kvq.h)."""
    _check(lib.attn_decode_append(ctypes.byref(layer), _ptr(seqs), n_seqs, _ptr(pos), max_pos, _ptr(q_raw),
                                  _ptr(k_raw), _ptr(v_raw), _ptr(q_norm_w), _ptr(k_norm_w), _ptr(out),
                                  int(out_is_f32), _ptr(q_prepped), _ptr(kv_prepped), _ptr(workspace),
                                  workspace_bytes, _stream(stream)))


def attn_prefill_append(layer: KvqLayer, seqs, n_seqs, row_offsets, start_pos, n_rows, max_rows_per_seq, q_raw,
                        k_raw, v_raw, q_norm_w, k_norm_w, out, out_is_f32, q_prepped, kv_prepped, workspace,
                        workspace_bytes, stream=None):
    """kv_quant_append of a chunk's rows, then attn_prefill_chunk, in one call
    (see include/kvq.h)."""
    _check(lib.attn_prefill_append(ctypes.byref(layer), _ptr(seqs), n_seqs, _ptr(row_offsets), _ptr(start_pos),
                                   n_rows, max_rows_per_seq, _ptr(q_raw), _ptr(k_raw), _ptr(v_raw),
                                   _ptr(q_norm_w), _ptr(k_norm_w), _ptr(out), int(out_is_f32), _ptr(q_prepped),
                                   _ptr(kv_prepped), _ptr(workspace), workspace_bytes, _stream(stream)))


def attn_train_donor_forward(layer: KvqLayer, n_blocks, block_offsets, n_rows, max_block_rows, q_raw, k_raw,
                             v_raw, q_norm_w, k_norm_w, k_hat, v_hat, out, out_is_f32, q_prepped, workspace,
                             workspace_bytes, stream=None):
    """kvq_train_kv_prep, then attn_train_forward, in one call (see include/kvq.h)."""
    _check(lib.attn_train_donor_forward(ctypes.byref(layer), n_blocks, _ptr(block_offsets), n_rows,
                                        max_block_rows, _ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _ptr(q_norm_w),
                                        _ptr(k_norm_w), _ptr(k_hat), _ptr(v_hat), _ptr(out), int(out_is_f32),
                                        _ptr(q_prepped), _ptr(workspace), workspace_bytes, _stream(stream)))


def attn_decode_static(layer: KvqLayer, seqs, n_seqs, pos, max_pos, q_raw, q_norm_w, out, out_is_f32,
                       q_prepped=None, stream=None):
    """attn_decode with the library's static scratch instead of a workspace
    (for callers that cannot allocate device memory; see include/kvq.h)."""
    _check(lib.attn_decode_static(ctypes.byref(layer), _ptr(seqs), n_seqs, _ptr(pos), max_pos, _ptr(q_raw),
                                  _ptr(q_norm_w), _ptr(out), int(out_is_f32), _ptr(q_prepped),
                                  _stream(stream)))


KVQ_STATIC_SCRATCH_BYTES = 16 << 20


def kvq_static_status(status, stream=None):
    """Copy the device status word of the latest attn_decode_static call into
    `status` (one uint32 of host or device memory: a numpy array, a torch
    tensor or an address); read it after the stream synchronizes."""
    if hasattr(status, "ctypes") and hasattr(status, "dtype"):          # numpy array
        addr = status.ctypes.data
    else:
        addr = _ptr(status)
    _check(lib.kvq_static_status(addr, _stream(stream)))


def attn_decode_workspace_bytes(layer: KvqLayer, n_seqs, max_pos) -> int:
    return lib.attn_decode_workspace_bytes(ctypes.byref(layer), n_seqs, max_pos)


def attn_prefill_chunk(layer: KvqLayer, seqs, n_seqs, row_offsets, start_pos, n_rows, max_rows_per_seq,
                       q_raw, q_norm_w, out, out_is_f32, q_prepped, workspace, workspace_bytes,
                       stream=None):
    _check(lib.attn_prefill_chunk(ctypes.byref(layer), _ptr(seqs), n_seqs, _ptr(row_offsets),
                                  _ptr(start_pos), n_rows, max_rows_per_seq, _ptr(q_raw),
                                  _ptr(q_norm_w), _ptr(out), int(out_is_f32), _ptr(q_prepped),
                                  _ptr(workspace), workspace_bytes, _stream(stream)))


def attn_prefill_workspace_bytes(layer: KvqLayer, n_seqs, n_rows, max_rows_per_seq) -> int:
    return lib.attn_prefill_workspace_bytes(ctypes.byref(layer), n_seqs, n_rows, max_rows_per_seq)


def kvq_train_kv_prep(layer: KvqLayer, n_blocks, block_offsets, n_rows, k_raw, v_raw, k_norm_w, k_hat, v_hat,
                      stream=None):
    """A donor layer's plain keys and values of a training pass (see include/kvq.h)."""
    _check(lib.kvq_train_kv_prep(ctypes.byref(layer), n_blocks, _ptr(block_offsets), n_rows, _ptr(k_raw),
                                 _ptr(v_raw), _ptr(k_norm_w), _ptr(k_hat), _ptr(v_hat), _stream(stream)))


def attn_train_forward(layer: KvqLayer, n_blocks, block_offsets, n_rows, max_block_rows, q_raw, q_norm_w,
                       k_hat, v_hat, out, out_is_f32, q_prepped, workspace, workspace_bytes, stream=None):
    """The training forward's read under a prefix-shared layout (see include/kvq.h)."""
    _check(lib.attn_train_forward(ctypes.byref(layer), n_blocks, _ptr(block_offsets), n_rows, max_block_rows,
                                  _ptr(q_raw), _ptr(q_norm_w), _ptr(k_hat), _ptr(v_hat), _ptr(out),
                                  int(out_is_f32), _ptr(q_prepped), _ptr(workspace), workspace_bytes,
                                  _stream(stream)))


def attn_train_workspace_bytes(layer: KvqLayer, n_rows) -> int:
    return lib.attn_train_workspace_bytes(ctypes.byref(layer), n_rows)


def attn_group(phase, seqs, n_seqs, row_offsets, pos, n_rows, max_pos, max_rows_per_seq, q_raw, out,
               q_prepped, workspace, workspace_bytes) -> KvqAttnGroup:
    """One group of attn_mixed (see include/kvq.h for the fields)."""
    return KvqAttnGroup(int(phase), _ptr(seqs), int(n_seqs), _ptr(row_offsets), _ptr(pos), int(n_rows),
                        int(max_pos), int(max_rows_per_seq), _ptr(q_raw), _ptr(out), _ptr(q_prepped),
                        _ptr(workspace), int(workspace_bytes))


def attn_mixed(layer: KvqLayer, groups, q_norm_w, out_is_f32, stream=None):
    arr = (KvqAttnGroup * max(1, len(groups)))(*groups)
    _check(lib.attn_mixed(ctypes.byref(layer), arr, len(groups), _ptr(q_norm_w), int(out_is_f32),
                          _stream(stream)))


def attn_mixed_schedule(layer: KvqLayer, groups, q_norm_w, out_is_f32) -> int:
    """Bit i set: group i of this attn_mixed call would run in the grouped
    decode-kernel launch (see include/kvq.h).  Host only."""
    arr = (KvqAttnGroup * max(1, len(groups)))(*groups)
    mask = ctypes.c_uint32(0)
    _check(lib.attn_mixed_schedule(ctypes.byref(layer), arr, len(groups), _ptr(q_norm_w), int(out_is_f32),
                                   ctypes.byref(mask)))
    return mask.value


def kvq_selftest_wait_timeout(status, limit_ns, stream=None):
    """Run the kernels' bounded wait on an mbarrier nothing completes (see
    include/kvq.h); bit 1 of the device uint32 `status` is set when it gives up."""
    _check(lib.kvq_selftest_wait_timeout(_ptr(status), int(limit_ns), _stream(stream)))


def kvq_profile_next_read(start_event, stop_event):
    """The next attention-reading call of this thread records the two events
    (torch.cuda.Event with timing, already created, or raw cudaEvent_t
    handles) around its attention kernel (see include/kvq.h)."""
    def handle(e):
        return None if e is None else int(getattr(e, "cuda_event", e))
    _check(lib.kvq_profile_next_read(handle(start_event), handle(stop_event)))


def kvq_status_string(status: int) -> str:
    return lib.kvq_status_string(status).decode()


def kvq_last_error() -> str:
    return lib.kvq_last_error().decode()


def kvq_version() -> int:
    return lib.kvq_version()


from .cache import LayerCaches  # noqa: E402,F401  (torch device memory for caches)
