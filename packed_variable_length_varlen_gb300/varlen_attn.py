"""Python binding of libvarlen_attn (the C ABI in include/varlen_attn.h).

Argument marshalling only: torch tensors become device pointers and int64
(row, head) strides, streams become cudaStream_t handles.  Every step of the
computation runs in the library's CUDA kernels; there is no fallback.  If the
library is missing or cannot be loaded, importing this module raises.

The raw entry points keep the C names (``varlen_attn_fwd`` ...) and return
the C status code.  ``attention_fwd`` / ``attention_bwd`` are conveniences
that allocate outputs / workspace with torch on the inputs' device and raise
``VarlenError`` on a non-zero status.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

VARLEN_OK = 0
VARLEN_ERR_NULL = -1
VARLEN_ERR_SHAPE = -2
VARLEN_ERR_HEAD_DIM = -3
VARLEN_ERR_ALIGN = -4
VARLEN_ERR_STRIDE = -5
VARLEN_ERR_WORKSPACE = -6
VARLEN_ERR_CUDA = -7
VARLEN_ERR_TIMEOUT = -8
VARLEN_ERR_DEVICE_BOUNDS = -9
VARLEN_ERR_ARCH = -10


class VarlenStride(ctypes.Structure):
    _fields_ = [("row", ctypes.c_int64), ("head", ctypes.c_int64)]


class VarlenDenseStride(ctypes.Structure):
    """Batch, row and head strides of one [batch, seqlen, H, D] tensor, in elements."""
    _fields_ = [("batch", ctypes.c_int64), ("row", ctypes.c_int64), ("head", ctypes.c_int64)]


class VarlenError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = "%s failed: %d (%s)" % (where, status, varlen_attn_status_string(status))
        if status == VARLEN_ERR_CUDA:
            msg += ": " + varlen_attn_last_cuda_error()
        super().__init__(msg)
        self.status = status


def _load() -> ctypes.CDLL:
    path = os.environ.get("VARLEN_ATTN_LIB", _build.LIB)
    if not os.path.exists(path):
        raise ImportError("libvarlen_attn not built at %s: run __graft_entry__.build() or "
                          "python -m packed_variable_length_varlen_gb300.build" % path)
    lib = ctypes.CDLL(path)
    S = VarlenStride
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.varlen_attn_fwd.restype = ctypes.c_int
    lib.varlen_attn_fwd.argtypes = [vp, S, vp, S, vp, S, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32,
                                    vp, S, vp, vp]
    lib.varlen_attn_bwd_workspace_size.restype = sz
    lib.varlen_attn_bwd_workspace_size.argtypes = [i32, i32, i32, i32]
    lib.varlen_attn_bwd.restype = ctypes.c_int
    lib.varlen_attn_bwd.argtypes = [vp, S, vp, S, vp, S, vp, S, vp, S, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                    i32, f32, vp, S, vp, S, vp, S, vp, sz, vp]
    lib.varlen_attn_fwd_causal.restype = ctypes.c_int
    lib.varlen_attn_fwd_causal.argtypes = lib.varlen_attn_fwd.argtypes
    lib.varlen_attn_bwd_causal.restype = ctypes.c_int
    lib.varlen_attn_bwd_causal.argtypes = lib.varlen_attn_bwd.argtypes
    lib.varlen_attn_fwd_window.restype = ctypes.c_int
    lib.varlen_attn_fwd_window.argtypes = [vp, S, vp, S, vp, S, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32,
                                           i32, i32, vp, S, vp, vp]
    lib.varlen_attn_bwd_window.restype = ctypes.c_int
    lib.varlen_attn_bwd_window.argtypes = [vp, S, vp, S, vp, S, vp, S, vp, S, vp, vp, vp, i32, i32, i32, i32, i32,
                                           i32, i32, f32, i32, i32, vp, S, vp, S, vp, S, vp, sz, vp]
    lib.varlen_attn_bwd_deterministic.restype = ctypes.c_int
    lib.varlen_attn_bwd_deterministic.argtypes = lib.varlen_attn_bwd_window.argtypes
    lib.varlen_attn_fwd_fp8_workspace_size.restype = sz
    lib.varlen_attn_fwd_fp8_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    lib.varlen_attn_fwd_fp8_workspace_layout.restype = ctypes.c_int
    lib.varlen_attn_fwd_fp8_workspace_layout.argtypes = [i32, i32, i32, i32, i32, vp, vp]
    lib.varlen_attn_fwd_fp8.restype = ctypes.c_int
    lib.varlen_attn_fwd_fp8.argtypes = [vp, S, vp, S, vp, S, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32, vp, S,
                                        vp, vp, sz, vp]
    lib.varlen_attn_fwd_fp8_window.restype = ctypes.c_int
    lib.varlen_attn_fwd_fp8_window.argtypes = [vp, S, vp, S, vp, S, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32,
                                               i32, i32, vp, S, vp, vp, sz, vp]
    DS = VarlenDenseStride
    lib.varlen_attn_fwd_fp8_dense_workspace_size.restype = sz
    lib.varlen_attn_fwd_fp8_dense_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    lib.varlen_attn_fwd_fp8_dense.restype = ctypes.c_int
    lib.varlen_attn_fwd_fp8_dense.argtypes = [vp, DS, vp, DS, vp, DS, i32, i32, i32, i32, i32, f32, i32, vp, DS, vp,
                                              vp, sz, vp]
    lib.varlen_attn_fwd_dense.restype = ctypes.c_int
    lib.varlen_attn_fwd_dense.argtypes = [vp, DS, vp, DS, vp, DS, i32, i32, i32, i32, i32, f32, i32, vp, DS, vp, vp]
    lib.varlen_attn_bwd_dense_workspace_size.restype = sz
    lib.varlen_attn_bwd_dense_workspace_size.argtypes = [i32, i32, i32, i32]
    lib.varlen_attn_bwd_dense.restype = ctypes.c_int
    lib.varlen_attn_bwd_dense.argtypes = [vp, DS, vp, DS, vp, DS, vp, DS, vp, DS, vp, i32, i32, i32, i32, i32, f32,
                                          i32, vp, DS, vp, DS, vp, DS, vp, sz, vp]
    lib.varlen_attn_bwd_noalloc.restype = ctypes.c_int
    lib.varlen_attn_bwd_noalloc.argtypes = [vp, S, vp, S, vp, S, vp, S, vp, S, vp, vp, vp, i32, i32, i32, i32, i32,
                                            i32, i32, f32, vp, S, vp, S, vp, S, vp]
    lib.varlen_attn_bwd_noalloc_scratch_bytes.restype = sz
    lib.varlen_attn_bwd_noalloc_scratch_bytes.argtypes = []
    lib.varlen_attn_debug_noalloc_scratch.restype = ctypes.c_int
    lib.varlen_attn_debug_noalloc_scratch.argtypes = [vp, vp]
    lib.varlen_attn_bounds_checked.restype = ctypes.c_int
    lib.varlen_attn_bounds_checked.argtypes = []
    lib.varlen_attn_debug_set_span_slack.restype = ctypes.c_int
    lib.varlen_attn_debug_set_span_slack.argtypes = [i64]
    lib.varlen_attn_debug_skip_load.restype = ctypes.c_int
    lib.varlen_attn_debug_skip_load.argtypes = [ctypes.c_int, i64]
    lib.varlen_attn_get_device_status.restype = ctypes.c_int
    lib.varlen_attn_get_device_status.argtypes = [vp]
    lib.varlen_attn_status_string.restype = ctypes.c_char_p
    lib.varlen_attn_status_string.argtypes = [ctypes.c_int]
    lib.varlen_attn_last_cuda_error.restype = ctypes.c_char_p
    lib.varlen_attn_last_cuda_error.argtypes = []
    lib.varlen_attn_tile_count.restype = i64
    lib.varlen_attn_tile_count.argtypes = [vp, i32, i32, i32, i32]
    lib.varlen_attn_debug_schedule.restype = ctypes.c_int
    lib.varlen_attn_debug_schedule.argtypes = [vp, i32, i32, i32, i32, i32, vp, i64, vp]
    lib.varlen_attn_selftest_wait_timeout.restype = ctypes.c_int
    lib.varlen_attn_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
    lib.varlen_attn_debug_mma_cycles.restype = ctypes.c_int
    lib.varlen_attn_debug_mma_cycles.argtypes = [i32, i32, i32, vp, vp]
    lib.varlen_attn_debug_set_phase_events.restype = ctypes.c_int
    lib.varlen_attn_debug_set_phase_events.argtypes = [vp, ctypes.c_int]
    lib.varlen_attn_num_sms.restype = ctypes.c_int
    lib.varlen_attn_num_sms.argtypes = []
    return lib


LIB = _load()
LIB_PATH = LIB._name

EXPORTED = ("varlen_attn_fwd", "varlen_attn_bwd_workspace_size", "varlen_attn_bwd",
            "varlen_attn_get_device_status", "varlen_attn_status_string", "varlen_attn_tile_count",
            "varlen_attn_debug_schedule", "varlen_attn_selftest_wait_timeout", "varlen_attn_num_sms",
            "varlen_attn_debug_set_phase_events", "varlen_attn_bwd_noalloc", "varlen_attn_last_cuda_error",
            "varlen_attn_fwd_causal", "varlen_attn_bwd_causal", "varlen_attn_fwd_dense",
            "varlen_attn_bwd_dense_workspace_size", "varlen_attn_bwd_dense", "varlen_attn_fwd_window",
            "varlen_attn_bwd_window", "varlen_attn_bwd_deterministic", "varlen_attn_fwd_fp8_workspace_size",
            "varlen_attn_fwd_fp8_workspace_layout", "varlen_attn_fwd_fp8", "varlen_attn_bwd_noalloc_scratch_bytes",
            "varlen_attn_debug_noalloc_scratch", "varlen_attn_bounds_checked", "varlen_attn_debug_set_span_slack",
            "varlen_attn_debug_skip_load", "varlen_attn_debug_mma_cycles", "varlen_attn_fwd_fp8_window",
            "varlen_attn_fwd_fp8_dense_workspace_size", "varlen_attn_fwd_fp8_dense")

# Size of the fixed device array varlen_attn_bwd_noalloc uses as scratch, as
# compiled into the library.
NOALLOC_SCRATCH_BYTES = int(LIB.varlen_attn_bwd_noalloc_scratch_bytes())


# ---------------------------------------------------------------- marshalling

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stride(t) -> VarlenStride:
    if t is None:
        return VarlenStride(0, 0)
    if t.dim() != 3 or t.stride(2) != 1:
        raise ValueError("NHD tensors must be [rows, heads, head_dim] with unit innermost stride")
    return VarlenStride(t.stride(0), t.stride(1))


def _dstride(t) -> VarlenDenseStride:
    if t is None:
        return VarlenDenseStride(0, 0, 0)
    if t.dim() != 4 or t.stride(3) != 1:
        raise ValueError("dense tensors must be [batch, seqlen, heads, head_dim] with unit innermost stride")
    return VarlenDenseStride(t.stride(0), t.stride(1), t.stride(2))


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    return ctypes.c_void_p(int(stream))


# ---------------------------------------------------------------- raw ABI

def _band(causal, window):
    """(left, right) of the window entry points for `causal` / `window`
    (causal sets right = 0), or None when neither masks anything."""
    left, right = int(window[0]), int(window[1])
    if causal:
        right = 0
    if left < 0 and right < 0:
        return None
    return max(left, -1), max(right, -1)


def varlen_attn_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, num_heads, head_dim,
                    max_seqlen_q, max_seqlen_k, scale, out, lse, stream=None, causal=False, window=(-1, -1)) -> int:
    band = _band(causal, window)
    head = (_ptr(q), _stride(q), _ptr(k), _stride(k), _ptr(v), _stride(v), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
            batch, total_q, total_k, num_heads, head_dim, max_seqlen_q, max_seqlen_k, scale)
    tail = (_ptr(out), _stride(out), _ptr(lse), _stream(stream))
    if band is None:
        return LIB.varlen_attn_fwd(*head, *tail)
    if band == (-1, 0):
        return LIB.varlen_attn_fwd_causal(*head, *tail)
    return LIB.varlen_attn_fwd_window(*head, *band, *tail)


def varlen_attn_fwd_window(q, k, v, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, num_heads, head_dim,
                           max_seqlen_q, max_seqlen_k, scale, window_left, window_right, out, lse,
                           stream=None) -> int:
    return LIB.varlen_attn_fwd_window(_ptr(q), _stride(q), _ptr(k), _stride(k), _ptr(v), _stride(v),
                                      _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), batch, total_q, total_k, num_heads,
                                      head_dim, max_seqlen_q, max_seqlen_k, scale, window_left, window_right,
                                      _ptr(out), _stride(out), _ptr(lse), _stream(stream))


def varlen_attn_fwd_causal(q, k, v, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, num_heads, head_dim,
                           max_seqlen_q, max_seqlen_k, scale, out, lse, stream=None) -> int:
    return varlen_attn_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, num_heads, head_dim,
                           max_seqlen_q, max_seqlen_k, scale, out, lse, stream, causal=True)


def varlen_attn_bwd_workspace_size(batch, total_q, num_heads, head_dim) -> int:
    return int(LIB.varlen_attn_bwd_workspace_size(batch, total_q, num_heads, head_dim))


def varlen_attn_bwd(q, k, v, out, dout, lse, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, num_heads,
                    head_dim, max_seqlen_q, max_seqlen_k, scale, dq, dk, dv, workspace, workspace_bytes,
                    stream=None, causal=False, window=(-1, -1), deterministic=False) -> int:
    band = _band(causal, window)
    head = (_ptr(q), _stride(q), _ptr(k), _stride(k), _ptr(v), _stride(v), _ptr(out), _stride(out), _ptr(dout),
            _stride(dout), _ptr(lse), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), batch, total_q, total_k, num_heads,
            head_dim, max_seqlen_q, max_seqlen_k, scale)
    tail = (_ptr(dq), _stride(dq), _ptr(dk), _stride(dk), _ptr(dv), _stride(dv), _ptr(workspace), workspace_bytes,
            _stream(stream))
    if deterministic:
        return LIB.varlen_attn_bwd_deterministic(*head, *(band or (-1, -1)), *tail)
    if band is None:
        return LIB.varlen_attn_bwd(*head, *tail)
    if band == (-1, 0):
        return LIB.varlen_attn_bwd_causal(*head, *tail)
    return LIB.varlen_attn_bwd_window(*head, *band, *tail)


def varlen_attn_bwd_window(q, k, v, out, dout, lse, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k,
                           num_heads, head_dim, max_seqlen_q, max_seqlen_k, scale, window_left, window_right, dq, dk,
                           dv, workspace, workspace_bytes, stream=None) -> int:
    return LIB.varlen_attn_bwd_window(_ptr(q), _stride(q), _ptr(k), _stride(k), _ptr(v), _stride(v), _ptr(out),
                                      _stride(out), _ptr(dout), _stride(dout), _ptr(lse), _ptr(cu_seqlens_q),
                                      _ptr(cu_seqlens_k), batch, total_q, total_k, num_heads, head_dim,
                                      max_seqlen_q, max_seqlen_k, scale, window_left, window_right, _ptr(dq),
                                      _stride(dq), _ptr(dk), _stride(dk), _ptr(dv), _stride(dv), _ptr(workspace),
                                      workspace_bytes, _stream(stream))


def varlen_attn_bwd_causal(q, k, v, out, dout, lse, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k,
                           num_heads, head_dim, max_seqlen_q, max_seqlen_k, scale, dq, dk, dv, workspace,
                           workspace_bytes, stream=None) -> int:
    return varlen_attn_bwd(q, k, v, out, dout, lse, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k,
                           num_heads, head_dim, max_seqlen_q, max_seqlen_k, scale, dq, dk, dv, workspace,
                           workspace_bytes, stream, causal=True)


def varlen_attn_fwd_fp8_workspace_size(batch, total_q, total_k, num_heads, head_dim) -> int:
    return int(LIB.varlen_attn_fwd_fp8_workspace_size(batch, total_q, total_k, num_heads, head_dim))


def varlen_attn_fwd_fp8_workspace_layout(batch, total_q, total_k, num_heads, head_dim):
    """(status, [amax, q codes, k codes, V^T codes] byte offsets, V^T row length)."""
    off = (ctypes.c_size_t * 4)()
    cols = ctypes.c_int64()
    st = LIB.varlen_attn_fwd_fp8_workspace_layout(batch, total_q, total_k, num_heads, head_dim,
                                                  ctypes.addressof(off), ctypes.addressof(cols))
    return st, list(off), int(cols.value)


def varlen_attn_fwd_fp8(q, k, v, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, num_heads, head_dim,
                        max_seqlen_q, max_seqlen_k, scale, out, lse, workspace, workspace_bytes, stream=None,
                        causal=False, window=(-1, -1)) -> int:
    band = _band(causal, window)
    head = (_ptr(q), _stride(q), _ptr(k), _stride(k), _ptr(v), _stride(v), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
            batch, total_q, total_k, num_heads, head_dim, max_seqlen_q, max_seqlen_k, scale)
    tail = (_ptr(out), _stride(out), _ptr(lse), _ptr(workspace), workspace_bytes, _stream(stream))
    if band is None:
        return LIB.varlen_attn_fwd_fp8(*head, *tail)
    return LIB.varlen_attn_fwd_fp8_window(*head, *band, *tail)


def varlen_attn_fwd_fp8_window(q, k, v, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, num_heads, head_dim,
                               max_seqlen_q, max_seqlen_k, scale, window_left, window_right, out, lse, workspace,
                               workspace_bytes, stream=None) -> int:
    return LIB.varlen_attn_fwd_fp8_window(_ptr(q), _stride(q), _ptr(k), _stride(k), _ptr(v), _stride(v),
                                          _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), batch, total_q, total_k, num_heads,
                                          head_dim, max_seqlen_q, max_seqlen_k, scale, window_left, window_right,
                                          _ptr(out), _stride(out), _ptr(lse), _ptr(workspace), workspace_bytes,
                                          _stream(stream))


def varlen_attn_fwd_fp8_dense_workspace_size(batch, seqlen_q, seqlen_k, num_heads, head_dim) -> int:
    return int(LIB.varlen_attn_fwd_fp8_dense_workspace_size(batch, seqlen_q, seqlen_k, num_heads, head_dim))


def varlen_attn_fwd_fp8_dense(q, k, v, batch, seqlen_q, seqlen_k, num_heads, head_dim, scale, causal, out, lse,
                              workspace, workspace_bytes, stream=None) -> int:
    return LIB.varlen_attn_fwd_fp8_dense(_ptr(q), _dstride(q), _ptr(k), _dstride(k), _ptr(v), _dstride(v), batch,
                                         seqlen_q, seqlen_k, num_heads, head_dim, scale, int(bool(causal)), _ptr(out),
                                         _dstride(out), _ptr(lse), _ptr(workspace), workspace_bytes,
                                         _stream(stream))


def varlen_attn_fwd_dense(q, k, v, batch, seqlen_q, seqlen_k, num_heads, head_dim, scale, causal, out, lse,
                          stream=None) -> int:
    return LIB.varlen_attn_fwd_dense(_ptr(q), _dstride(q), _ptr(k), _dstride(k), _ptr(v), _dstride(v), batch,
                                     seqlen_q, seqlen_k, num_heads, head_dim, scale, int(bool(causal)), _ptr(out),
                                     _dstride(out), _ptr(lse), _stream(stream))


def varlen_attn_bwd_dense_workspace_size(batch, seqlen_q, num_heads, head_dim) -> int:
    return int(LIB.varlen_attn_bwd_dense_workspace_size(batch, seqlen_q, num_heads, head_dim))


def varlen_attn_bwd_dense(q, k, v, out, dout, lse, batch, seqlen_q, seqlen_k, num_heads, head_dim, scale, causal,
                          dq, dk, dv, workspace, workspace_bytes, stream=None) -> int:
    return LIB.varlen_attn_bwd_dense(_ptr(q), _dstride(q), _ptr(k), _dstride(k), _ptr(v), _dstride(v), _ptr(out),
                                     _dstride(out), _ptr(dout), _dstride(dout), _ptr(lse), batch, seqlen_q, seqlen_k,
                                     num_heads, head_dim, scale, int(bool(causal)), _ptr(dq), _dstride(dq), _ptr(dk),
                                     _dstride(dk), _ptr(dv), _dstride(dv), _ptr(workspace), workspace_bytes,
                                     _stream(stream))


def varlen_attn_bwd_noalloc(q, k, v, out, dout, lse, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k,
                            num_heads, head_dim, max_seqlen_q, max_seqlen_k, scale, dq, dk, dv, stream=None) -> int:
    """The backward for callers that cannot allocate device memory: scratch
    comes from a fixed library-owned device array (see the C header)."""
    return LIB.varlen_attn_bwd_noalloc(_ptr(q), _stride(q), _ptr(k), _stride(k), _ptr(v), _stride(v), _ptr(out),
                                       _stride(out), _ptr(dout), _stride(dout), _ptr(lse), _ptr(cu_seqlens_q),
                                       _ptr(cu_seqlens_k), batch, total_q, total_k, num_heads, head_dim,
                                       max_seqlen_q, max_seqlen_k, scale, _ptr(dq), _stride(dq), _ptr(dk),
                                       _stride(dk), _ptr(dv), _stride(dv), _stream(stream))


def varlen_attn_debug_noalloc_scratch():
    """(status, scratch device address, context id) that the next
    varlen_attn_bwd_noalloc call on this thread would use; launches nothing."""
    addr = ctypes.c_void_p(0)
    ctx = ctypes.c_ulonglong(0)
    st = LIB.varlen_attn_debug_noalloc_scratch(ctypes.byref(addr), ctypes.byref(ctx))
    return st, int(addr.value or 0), int(ctx.value)


def varlen_attn_bounds_checked() -> bool:
    """True for a library built with device-side bounds checks."""
    return bool(LIB.varlen_attn_bounds_checked())


def varlen_attn_debug_set_span_slack(nbytes: int) -> int:
    return LIB.varlen_attn_debug_set_span_slack(int(nbytes))


def varlen_attn_debug_skip_load(which: int, n: int) -> int:
    return LIB.varlen_attn_debug_skip_load(int(which), int(n))


def varlen_attn_get_device_status(stream=None) -> int:
    return LIB.varlen_attn_get_device_status(_stream(stream))


def varlen_attn_status_string(status: int) -> str:
    return LIB.varlen_attn_status_string(status).decode()


def varlen_attn_last_cuda_error() -> str:
    return LIB.varlen_attn_last_cuda_error().decode()


def varlen_attn_tile_count(cu_seqlens_host, batch, total, num_heads, tile) -> int:
    cu = torch.as_tensor(cu_seqlens_host, dtype=torch.int32).contiguous()
    return int(LIB.varlen_attn_tile_count(ctypes.c_void_p(cu.data_ptr()), batch, total, num_heads, tile))


def varlen_attn_debug_schedule(cu_seqlens, batch, total, num_heads, tile, grid, out_records, max_records,
                               stream=None) -> int:
    return LIB.varlen_attn_debug_schedule(_ptr(cu_seqlens), batch, total, num_heads, tile, grid,
                                          _ptr(out_records), max_records, _stream(stream))


def varlen_attn_selftest_wait_timeout(budget_ns: int, stream=None) -> int:
    return LIB.varlen_attn_selftest_wait_timeout(budget_ns, _stream(stream))


def varlen_attn_debug_mma_cycles(n_mma, n_cols, mode, cycles, stream=None) -> int:
    """cycles: a CUDA int64 tensor (one element) that receives the count."""
    return LIB.varlen_attn_debug_mma_cycles(n_mma, n_cols, mode, _ptr(cycles), _stream(stream))


_PHASE_KEEP = None


def varlen_attn_debug_set_phase_events(events) -> int:
    """events: four torch.cuda.Event(enable_timing=True) objects, or None."""
    global _PHASE_KEEP
    if not events:
        _PHASE_KEEP = None
        return LIB.varlen_attn_debug_set_phase_events(None, 0)
    for e in events:
        e.record()  # materialise the handle on the current device
    arr = (ctypes.c_void_p * 4)(*[e.cuda_event for e in events])
    _PHASE_KEEP = (events, arr)
    return LIB.varlen_attn_debug_set_phase_events(arr, 4)


def varlen_attn_num_sms() -> int:
    return LIB.varlen_attn_num_sms()


# ---------------------------------------------------------------- conveniences

def _check(status, where):
    if status != VARLEN_OK:
        raise VarlenError(status, where)


def attention_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q=0, max_seqlen_k=0, scale=None,
                  out=None, lse=None, stream=None, causal=False, window=(-1, -1)):
    """O and LSE for packed q/k/v ([rows, H, D] bf16 on one CUDA device);
    `causal` / `window` = (left, right) select the masked entry points
    (causal sets right = 0; a negative side is unbounded)."""
    total_q, H, D = q.shape
    total_k = k.shape[0]
    batch = cu_seqlens_q.numel() - 1
    scale = float(D ** -0.5) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q, memory_format=torch.contiguous_format)
    if lse is None:
        lse = torch.empty(H, total_q, dtype=torch.float32, device=q.device)
    _check(varlen_attn_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, H, D, max_seqlen_q,
                           max_seqlen_k, scale, out, lse, stream, causal, window), "varlen_attn_fwd")
    return out, lse


def attention_fwd_fp8(q, k, v, cu_seqlens_q, cu_seqlens_k, scale=None, out=None, lse=None, workspace=None,
                      stream=None, causal=False, window=(-1, -1)):
    """E4M3 forward of packed bf16 q/k/v ([rows, H, 128]): quantised per
    (segment, head) into `workspace` (allocated when None), O in bf16 and
    LSE, optionally under a causal or sliding-window band.  Returns (out,
    lse, workspace)."""
    total_q, H, D = q.shape
    total_k = k.shape[0]
    batch = cu_seqlens_q.numel() - 1
    scale = float(D ** -0.5) if scale is None else float(scale)
    nbytes = varlen_attn_fwd_fp8_workspace_size(batch, total_q, total_k, H, D)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q, memory_format=torch.contiguous_format)
    if lse is None:
        lse = torch.empty(H, total_q, dtype=torch.float32, device=q.device)
    _check(varlen_attn_fwd_fp8(q, k, v, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, H, D, 0, 0, scale, out,
                               lse, workspace, workspace.numel(), stream, causal, window), "varlen_attn_fwd_fp8")
    return out, lse, workspace


def attention_bwd(q, k, v, out, dout, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q=0, max_seqlen_k=0,
                  scale=None, dq=None, dk=None, dv=None, workspace=None, stream=None, causal=False,
                  window=(-1, -1), deterministic=False):
    """dQ, dK, dV for the forward above (every operand keeps its strides)."""
    total_q, H, D = q.shape
    total_k = k.shape[0]
    batch = cu_seqlens_q.numel() - 1
    scale = float(D ** -0.5) if scale is None else float(scale)
    dq = torch.empty_like(q, memory_format=torch.contiguous_format) if dq is None else dq
    dk = torch.empty_like(k, memory_format=torch.contiguous_format) if dk is None else dk
    dv = torch.empty_like(v, memory_format=torch.contiguous_format) if dv is None else dv
    nbytes = varlen_attn_bwd_workspace_size(batch, total_q, H, D)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    _check(varlen_attn_bwd(q, k, v, out, dout, lse, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, H, D,
                           max_seqlen_q, max_seqlen_k, scale, dq, dk, dv, workspace, workspace.numel(), stream,
                           causal, window, deterministic), "varlen_attn_bwd")
    return dq, dk, dv


def attention_fwd_dense(q, k, v, scale=None, causal=False, out=None, lse=None, stream=None):
    """O and LSE for dense batched q [B, Sq, H, D], k / v [B, Sk, H, D] (bf16,
    one CUDA device); lse is [H, B * Sq]."""
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    scale = float(D ** -0.5) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q, memory_format=torch.contiguous_format)
    if lse is None:
        lse = torch.empty(H, B * Sq, dtype=torch.float32, device=q.device)
    _check(varlen_attn_fwd_dense(q, k, v, B, Sq, Sk, H, D, scale, causal, out, lse, stream), "varlen_attn_fwd_dense")
    return out, lse


def attention_fwd_fp8_dense(q, k, v, scale=None, causal=False, out=None, lse=None, workspace=None, stream=None):
    """E4M3 forward of dense batched bf16 q [B, Sq, H, 128], k / v
    [B, Sk, H, 128]: quantised per (batch entry, head) into `workspace`
    (allocated when None); returns (out, lse [H, B * Sq], workspace)."""
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    scale = float(D ** -0.5) if scale is None else float(scale)
    nbytes = varlen_attn_fwd_fp8_dense_workspace_size(B, Sq, Sk, H, D)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q, memory_format=torch.contiguous_format)
    if lse is None:
        lse = torch.empty(H, B * Sq, dtype=torch.float32, device=q.device)
    _check(varlen_attn_fwd_fp8_dense(q, k, v, B, Sq, Sk, H, D, scale, causal, out, lse, workspace,
                                     workspace.numel(), stream), "varlen_attn_fwd_fp8_dense")
    return out, lse, workspace


def attention_bwd_dense(q, k, v, out, dout, lse, scale=None, causal=False, dq=None, dk=None, dv=None,
                        workspace=None, stream=None):
    """dQ, dK, dV for attention_fwd_dense."""
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    scale = float(D ** -0.5) if scale is None else float(scale)
    dq = torch.empty_like(q, memory_format=torch.contiguous_format) if dq is None else dq
    dk = torch.empty_like(k, memory_format=torch.contiguous_format) if dk is None else dk
    dv = torch.empty_like(v, memory_format=torch.contiguous_format) if dv is None else dv
    nbytes = varlen_attn_bwd_dense_workspace_size(B, Sq, H, D)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    _check(varlen_attn_bwd_dense(q, k, v, out, dout, lse, B, Sq, Sk, H, D, scale, causal, dq, dk, dv, workspace,
                                 workspace.numel(), stream), "varlen_attn_bwd_dense")
    return dq, dk, dv
