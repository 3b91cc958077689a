"""Gated delta rule on GB300 (sm_103a): a thin Python binding of libgdr.so.

Every function here only marshals arguments into the C ABI declared in
include/gdr.h (same names); all arithmetic runs in the library's CUDA kernels.
PyTorch is used for device memory and streams only.  There is no CPU path:
if the compiled library is missing, every call raises.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

__all__ = [
    "GdrError", "gdr_dims", "lib", "library_path",
    "gdr_prefill_chunked", "gdr_prefill_workspace_bytes", "gdr_prefill_chunked_static",
    "gdr_prefill_segmented", "gdr_prefill_segmented_workspace_bytes", "gdr_prefill_segments_hint",
    "gdr_decode_step", "gdr_decode_step_overlapped", "gdr_decode_step_gated", "gdr_gated_rmsnorm",
    "gdr_prefill_with_decode",
    "gdr_verify_block", "gdr_verify_commit",
    "gdr_state_snapshot", "gdr_state_restore", "gdr_device_error", "gdr_selftest_wait_timeout", "gdr_status_string",
    "GDR_F32", "GDR_BF16", "GDR_FLAG_QK_L2NORM", "GDR_FLAG_BETA_LOGITS",
]

GDR_OK, GDR_ERR_INVALID_ARG, GDR_ERR_UNSUPPORTED, GDR_ERR_CUDA, GDR_ERR_DEVICE_TIMEOUT = range(5)
GDR_F32, GDR_BF16 = 0, 1
GDR_FLAG_QK_L2NORM, GDR_FLAG_BETA_LOGITS = 1, 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return os.path.join(_HERE, "libgdr.so")


class GdrError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {gdr_status_string(status)}")


class gdr_dims(ctypes.Structure):
    _fields_ = [
        ("h_qk", ctypes.c_int32), ("h_v", ctypes.c_int32),
        ("d_k", ctypes.c_int32), ("d_v", ctypes.c_int32),
        ("chunk", ctypes.c_int32), ("in_dtype", ctypes.c_int32),
        ("out_dtype", ctypes.c_int32), ("scale", ctypes.c_float),
        ("flags", ctypes.c_int32),
    ]


_P = ctypes.c_void_p
_SIGS = {
    "gdr_abi_version": ([], ctypes.c_int32),
    "gdr_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "gdr_prefill_workspace_bytes": ([ctypes.POINTER(gdr_dims), ctypes.c_int32, ctypes.c_int64],
                                    ctypes.c_size_t),
    "gdr_prefill_chunked": ([ctypes.POINTER(gdr_dims), ctypes.c_int32, _P, ctypes.c_int64,
                             _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P], ctypes.c_int),
    "gdr_prefill_chunked_static": ([ctypes.POINTER(gdr_dims), ctypes.c_int32, _P, ctypes.c_int64,
                                    _P, _P, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "gdr_prefill_static_workspace_capacity": ([], ctypes.c_size_t),
    "gdr_prefill_segmented": ([ctypes.POINTER(gdr_dims), ctypes.c_int32, _P, ctypes.c_int64,
                               _P, _P, _P, _P, _P, _P, _P, ctypes.c_int32, _P, ctypes.c_size_t, _P], ctypes.c_int),
    "gdr_prefill_segmented_workspace_bytes": ([ctypes.POINTER(gdr_dims), ctypes.c_int32, ctypes.c_int64,
                                               ctypes.c_int32], ctypes.c_size_t),
    "gdr_prefill_segments_hint": ([ctypes.POINTER(gdr_dims), ctypes.c_int32, ctypes.c_int64], ctypes.c_int32),
    "gdr_decode_step": ([ctypes.POINTER(gdr_dims), ctypes.c_int32, _P, _P, _P, _P, _P, _P, _P, _P],
                        ctypes.c_int),
    "gdr_decode_step_overlapped": ([ctypes.POINTER(gdr_dims), ctypes.c_int32, _P, _P, _P, _P, _P, _P, _P, _P],
                                   ctypes.c_int),
    "gdr_prefill_with_decode": ([ctypes.POINTER(gdr_dims), ctypes.c_int32, _P, ctypes.c_int64,
                                 _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, ctypes.c_int32,
                                 _P, _P, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "gdr_verify_block": ([ctypes.POINTER(gdr_dims), ctypes.c_int32, ctypes.c_int32,
                          _P, _P, _P, _P, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "gdr_verify_commit": ([ctypes.POINTER(gdr_dims), ctypes.c_int32, ctypes.c_int32,
                           _P, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "gdr_decode_step_gated": ([ctypes.POINTER(gdr_dims), ctypes.c_int32, _P, _P, _P, _P, _P, _P, _P, _P,
                               ctypes.c_float, _P, _P], ctypes.c_int),
    "gdr_gated_rmsnorm": ([ctypes.POINTER(gdr_dims), ctypes.c_int64, _P, _P, _P, ctypes.c_float, _P, _P],
                          ctypes.c_int),
    "gdr_state_snapshot": ([ctypes.POINTER(gdr_dims), ctypes.c_int32, _P, _P, _P], ctypes.c_int),
    "gdr_state_restore": ([ctypes.POINTER(gdr_dims), ctypes.c_int32, _P, _P, _P], ctypes.c_int),
    "gdr_device_error": ([_P, ctypes.POINTER(ctypes.c_int32)], ctypes.c_int),
    "gdr_selftest_wait_timeout": ([ctypes.c_int64, _P], ctypes.c_int),
}


def lib():
    """The loaded library (ctypes); raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise ImportError(
                    f"{path} is missing: build it with `python -m gated_deltanet_scan_gb300.build` "
                    "(there is no CPU fallback)")
            handle = ctypes.CDLL(path)
            for name, (argtypes, restype) in _SIGS.items():
                fn = getattr(handle, name)
                fn.argtypes = argtypes
                fn.restype = restype
            _lib = handle
    return _lib


def gdr_status_string(status: int) -> str:
    try:
        return lib().gdr_status_string(int(status)).decode()
    except ImportError:
        return f"gdr_status {status}"


def _check(status: int, where: str) -> None:
    if status != GDR_OK:
        raise GdrError(status, where)


# --- marshalling helpers (torch only for pointers, dtypes and streams) ----------

def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return GDR_BF16
    if t.dtype == torch.float32:
        return GDR_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream_handle(stream, device) -> Optional[int]:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def flags_of(qk_l2norm: bool = False, beta_logits: bool = False) -> int:
    return (GDR_FLAG_QK_L2NORM if qk_l2norm else 0) | (GDR_FLAG_BETA_LOGITS if beta_logits else 0)


def make_dims(q, v, o, chunk: int = 64, scale: float = 1.0, flags: int = 0) -> gdr_dims:
    """dims from q [T, H_qk, d_k], v [T, H_v, d_v] and o (its dtype is the output type)."""
    return gdr_dims(h_qk=q.shape[-2], h_v=v.shape[-2], d_k=q.shape[-1], d_v=v.shape[-1],
                    chunk=chunk, in_dtype=_dtype_code(q), out_dtype=_dtype_code(o),
                    scale=float(scale), flags=int(flags))


def gdr_prefill_workspace_bytes(q, v, o, n_seqs: int, t_total: int, *, chunk: int = 64,
                                scale: float = 1.0) -> int:
    """Device scratch bytes gdr_prefill_chunked needs (0 on the CUDA-core path)."""
    dims = make_dims(q, v, o, chunk, scale, 0)
    return int(lib().gdr_prefill_workspace_bytes(ctypes.byref(dims), int(n_seqs), int(t_total)))


def gdr_prefill_chunked(q, k, v, g, beta, state, o, cu_seqlens, *, chunk: int = 64,
                        scale: float = 1.0, qk_l2norm: bool = False, beta_logits: bool = False, t_total: Optional[int] = None, workspace=None,
                        stream=None) -> None:
    """Chunked prefill over packed sequences (see gdr_prefill_chunked in include/gdr.h).

    q, k [T, H_qk, d_k]; v [T, H_v, d_v]; g, beta [T, H_v] fp32;
    state [n, H_v, d_k, d_v] fp32 (in/out); o [T, H_v, d_v]; cu_seqlens int32 [n+1]
    on the device.  ``t_total`` defaults to q.shape[0].  ``workspace`` is a
    device tensor of at least gdr_prefill_workspace_bytes(...) bytes; when it is
    None, one is taken from torch's caching allocator for this call, on the
    stream the call runs on (``stream``), so that torch hands its memory to no
    other work before the call's kernels on that stream are done."""
    torch = _torch()
    dims = make_dims(q, v, o, chunk, scale, flags_of(qk_l2norm, beta_logits))
    n = cu_seqlens.shape[0] - 1
    T = q.shape[0] if t_total is None else int(t_total)
    need = int(lib().gdr_prefill_workspace_bytes(ctypes.byref(dims), n, T))
    if workspace is None and need > 0:
        # allocated while the call's stream is current: the caching allocator ties
        # the block to that stream, whatever stream is current in the caller
        s = stream if stream is not None else torch.cuda.current_stream(q.device)
        if isinstance(s, int):
            s = torch.cuda.ExternalStream(s, device=q.device)
        with torch.cuda.stream(s):
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _ptr(workspace) if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().gdr_prefill_chunked(
        ctypes.byref(dims), n, _ptr(cu_seqlens), T, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
        _ptr(beta), _ptr(state), _ptr(o), ws_ptr, ws_bytes, _stream_handle(stream, q.device))
    _check(st, "gdr_prefill_chunked")


def gdr_prefill_chunked_static(q, k, v, g, beta, state, o, cu_seqlens, *, chunk: int = 64,
                               scale: float = 1.0, qk_l2norm: bool = False, beta_logits: bool = False,
                               t_total: Optional[int] = None, stream=None) -> None:
    """gdr_prefill_chunked with the library's fixed scratch array instead of a
    workspace (nothing is allocated; see include/gdr.h for its size limit)."""
    dims = make_dims(q, v, o, chunk, scale, flags_of(qk_l2norm, beta_logits))
    n = cu_seqlens.shape[0] - 1
    T = q.shape[0] if t_total is None else int(t_total)
    st = lib().gdr_prefill_chunked_static(
        ctypes.byref(dims), n, _ptr(cu_seqlens), T, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
        _ptr(beta), _ptr(state), _ptr(o), _stream_handle(stream, q.device))
    _check(st, "gdr_prefill_chunked_static")


def gdr_prefill_segments_hint(q, v, o, n_seqs: int, t_total: int, *, chunk: int = 64, scale: float = 1.0) -> int:
    """Segments the two-level prefill would use on the current device (1: none)."""
    dims = make_dims(q, v, o, chunk, scale, 0)
    return int(lib().gdr_prefill_segments_hint(ctypes.byref(dims), int(n_seqs), int(t_total)))


def gdr_prefill_segmented_workspace_bytes(q, v, o, n_seqs: int, t_total: int, n_segments: int, *,
                                          chunk: int = 64, scale: float = 1.0) -> int:
    dims = make_dims(q, v, o, chunk, scale, 0)
    return int(lib().gdr_prefill_segmented_workspace_bytes(ctypes.byref(dims), int(n_seqs), int(t_total),
                                                           int(n_segments)))


def gdr_prefill_segmented(q, k, v, g, beta, state, o, cu_seqlens, n_segments: Optional[int] = None, *,
                          chunk: int = 64, scale: float = 1.0, qk_l2norm: bool = False, beta_logits: bool = False, t_total: Optional[int] = None, workspace=None,
                          stream=None) -> None:
    """Two-level (segment-parallel) prefill (see gdr_prefill_segmented in
    include/gdr.h): arguments as gdr_prefill_chunked; ``n_segments`` defaults to
    gdr_prefill_segments_hint.  Without ``workspace`` one is taken from torch's
    allocator on the call's stream."""
    torch = _torch()
    dims = make_dims(q, v, o, chunk, scale, flags_of(qk_l2norm, beta_logits))
    n = cu_seqlens.shape[0] - 1
    T = q.shape[0] if t_total is None else int(t_total)
    P = int(lib().gdr_prefill_segments_hint(ctypes.byref(dims), n, T)) if n_segments is None else int(n_segments)
    need = int(lib().gdr_prefill_segmented_workspace_bytes(ctypes.byref(dims), n, T, P))
    if workspace is None and need > 0:
        s = stream if stream is not None else torch.cuda.current_stream(q.device)
        if isinstance(s, int):
            s = torch.cuda.ExternalStream(s, device=q.device)
        with torch.cuda.stream(s):
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _ptr(workspace) if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().gdr_prefill_segmented(
        ctypes.byref(dims), n, _ptr(cu_seqlens), T, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state),
        _ptr(o), P, ws_ptr, ws_bytes, _stream_handle(stream, q.device))
    _check(st, "gdr_prefill_segmented")


def gdr_decode_step(q, k, v, g, beta, state, o, *, scale: float = 1.0, qk_l2norm: bool = False,
                    beta_logits: bool = False, stream=None) -> None:
    """One decode step for B sequences: q, k [B, H_qk, d]; v, o [B, H_v, d];
    g, beta [B, H_v]; state [B, H_v, d, d] updated in place."""
    dims = make_dims(q, v, o, 64, scale, flags_of(qk_l2norm, beta_logits))
    st = lib().gdr_decode_step(
        ctypes.byref(dims), q.shape[0], _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
        _ptr(state), _ptr(o), _stream_handle(stream, q.device))
    _check(st, "gdr_decode_step")


def gdr_prefill_with_decode(q, k, v, g, beta, state, o, cu_seqlens, dq, dk, dv, dg, dbeta, dstate, d_o, *,
                            scale: float = 1.0, qk_l2norm: bool = False, beta_logits: bool = False,
                            t_total: Optional[int] = None, workspace=None, stream=None) -> None:
    """A prefill (as gdr_prefill_chunked) and one decode step of another batch (as
    gdr_decode_step) in the same chunk-scan launch (see include/gdr.h)."""
    torch = _torch()
    dims = make_dims(q, v, o, 64, scale, flags_of(qk_l2norm, beta_logits))
    n = cu_seqlens.shape[0] - 1
    T = q.shape[0] if t_total is None else int(t_total)
    need = int(lib().gdr_prefill_workspace_bytes(ctypes.byref(dims), n, T))
    if workspace is None and need > 0:
        s = stream if stream is not None else torch.cuda.current_stream(q.device)
        if isinstance(s, int):
            s = torch.cuda.ExternalStream(s, device=q.device)
        with torch.cuda.stream(s):
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _ptr(workspace) if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().gdr_prefill_with_decode(
        ctypes.byref(dims), n, _ptr(cu_seqlens), T, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state),
        _ptr(o), ws_ptr, ws_bytes, dq.shape[0], _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(dstate),
        _ptr(d_o), _stream_handle(stream, q.device))
    _check(st, "gdr_prefill_with_decode")


def gdr_decode_step_overlapped(q, k, v, g, beta, state, o, *, scale: float = 1.0, qk_l2norm: bool = False,
                               beta_logits: bool = False, stream=None) -> None:
    """gdr_decode_step launched as a programmatic dependent of the kernel before it
    on the stream (see include/gdr.h): none of its inputs or states may be written
    by that kernel."""
    dims = make_dims(q, v, o, 64, scale, flags_of(qk_l2norm, beta_logits))
    st = lib().gdr_decode_step_overlapped(
        ctypes.byref(dims), q.shape[0], _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
        _ptr(state), _ptr(o), _stream_handle(stream, q.device))
    _check(st, "gdr_decode_step_overlapped")


RMSNORM_EPS = 1e-6  # the epsilon of the gated RMSNorm after the rule


def gdr_decode_step_gated(q, k, v, g, beta, state, z, weight, y, *, eps: float = RMSNORM_EPS, scale: float = 1.0,
                          qk_l2norm: bool = False, beta_logits: bool = False, stream=None) -> None:
    """gdr_decode_step with the gated RMSNorm fused: y = weight * o / sqrt(mean(o^2) + eps) * silu(z)
    per (sequence, V head) row; z [B, H_v, d] like v, weight [d] fp32, y like the output."""
    dims = make_dims(q, v, y, 64, scale, flags_of(qk_l2norm, beta_logits))
    st = lib().gdr_decode_step_gated(
        ctypes.byref(dims), q.shape[0], _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state), _ptr(z),
        _ptr(weight), float(eps), _ptr(y), _stream_handle(stream, q.device))
    _check(st, "gdr_decode_step_gated")


def gdr_gated_rmsnorm(o, z, weight, y, *, eps: float = RMSNORM_EPS, stream=None) -> None:
    """y = weight * o / sqrt(mean(o^2) + eps) * silu(z) over the last axis of o [..., d]
    (o and y fp32 or bf16, z fp32 or bf16, weight [d] fp32)."""
    d = o.shape[-1]
    rows = o.numel() // d
    dims = gdr_dims(h_qk=1, h_v=1, d_k=d, d_v=d, chunk=64, in_dtype=_dtype_code(z), out_dtype=_dtype_code(o),
                    scale=1.0, flags=0)
    if y.dtype != o.dtype:
        raise TypeError("y must have o's dtype")
    st = lib().gdr_gated_rmsnorm(ctypes.byref(dims), rows, _ptr(o), _ptr(z), _ptr(weight), float(eps), _ptr(y),
                                 _stream_handle(stream, o.device))
    _check(st, "gdr_gated_rmsnorm")


def gdr_verify_block(q, k, v, g, beta, state, snapshot, o, n_tok: int, *, deltas=None, scale: float = 1.0,
                     qk_l2norm: bool = False, beta_logits: bool = False, stream=None) -> None:
    """n_tok (<= 16) draft tokens per sequence from the current state; the incoming
    state is copied to ``snapshot``.  Token rows are [n_seqs * n_tok, ...].  With
    ``deltas`` (fp32, shaped like v) each token's correction is kept for
    gdr_verify_commit."""
    dims = make_dims(q, v, o, 16, scale, flags_of(qk_l2norm, beta_logits))
    n = state.shape[0]
    st = lib().gdr_verify_block(
        ctypes.byref(dims), n, int(n_tok), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
        _ptr(state), _ptr(snapshot), _ptr(o), _ptr(deltas), _stream_handle(stream, state.device))
    _check(st, "gdr_verify_block")


def gdr_verify_commit(k, g, deltas, snapshot, state, accepted, n_tok: int, *, qk_l2norm: bool = False,
                      stream=None) -> None:
    """State after the accepted prefix of a verify block: accepted (int32 device
    tensor [n_seqs]) tokens per sequence, from the block's ``deltas`` and the
    ``snapshot`` it took; writes ``state``."""
    n, hv, dk, dv = state.shape
    dims = gdr_dims(h_qk=k.shape[1], h_v=hv, d_k=dk, d_v=dv, chunk=16,
                    in_dtype=_dtype_code(k), out_dtype=GDR_F32, scale=1.0, flags=flags_of(qk_l2norm))
    st = lib().gdr_verify_commit(
        ctypes.byref(dims), n, int(n_tok), _ptr(accepted), _ptr(k), _ptr(g), _ptr(deltas),
        _ptr(snapshot), _ptr(state), _stream_handle(stream, state.device))
    _check(st, "gdr_verify_commit")


def _state_dims(state) -> gdr_dims:
    _, hv, dk, dv = state.shape
    return gdr_dims(h_qk=hv, h_v=hv, d_k=dk, d_v=dv, chunk=64, in_dtype=GDR_F32,
                    out_dtype=GDR_F32, scale=1.0)


def gdr_state_snapshot(state, snapshot, *, stream=None) -> None:
    dims = _state_dims(state)
    st = lib().gdr_state_snapshot(ctypes.byref(dims), state.shape[0], _ptr(state), _ptr(snapshot),
                                  _stream_handle(stream, state.device))
    _check(st, "gdr_state_snapshot")


def gdr_state_restore(snapshot, state, *, stream=None) -> None:
    dims = _state_dims(state)
    st = lib().gdr_state_restore(ctypes.byref(dims), state.shape[0], _ptr(snapshot), _ptr(state),
                                 _stream_handle(stream, state.device))
    _check(st, "gdr_state_restore")


def gdr_device_error(*, stream=None, device=None) -> int:
    """Synchronise the stream and return (and clear) the device error word."""
    code = ctypes.c_int32(0)
    _check(lib().gdr_device_error(_stream_handle(stream, device), ctypes.byref(code)), "gdr_device_error")
    return int(code.value)


def gdr_selftest_wait_timeout(limit_cycles: int, *, stream=None, device=None) -> None:
    """Launch the self-test block whose bounded wait on a barrier nothing arrives
    on gives up after limit_cycles SM clocks and records GDR_ERR_DEVICE_TIMEOUT."""
    _check(lib().gdr_selftest_wait_timeout(int(limit_cycles), _stream_handle(stream, device)),
           "gdr_selftest_wait_timeout")
