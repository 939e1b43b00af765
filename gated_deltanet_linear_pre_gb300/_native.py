"""ctypes binding of libgdn.so (the C ABI in include/gdn.h).

Argument marshalling only: every entry point checks that the torch tensors it
is handed have the dtype, device, shape and contiguity the ABI documents,
passes their device pointers and the current CUDA stream, and raises
``GdnError`` on a non-OK status.  All arithmetic runs in the library's CUDA
kernels; there is no other implementation behind these names.  If the
library has not been built the first call raises (build it with
``python -m gated_deltanet_linear_pre_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

_lock = threading.Lock()
_lib = None

_p = ctypes.c_void_p
_i32 = ctypes.c_int32
_sz = ctypes.c_size_t

STATUS = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED", 3: "GDN_ERR_ALIGNMENT",
          4: "GDN_ERR_WORKSPACE", 5: "GDN_ERR_CUDA", 6: "GDN_ERR_TIMEOUT"}


class GdnError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str):
        self.status = status
        super().__init__(f"{fn}: {STATUS.get(status, status)}: {detail}")


class gdn_dims(ctypes.Structure):
    _fields_ = [("hk", ctypes.c_int32), ("hv", ctypes.c_int32), ("dk", ctypes.c_int32),
                ("dv", ctypes.c_int32), ("eps", ctypes.c_float)]


def dims(hk: int = 16, hv: int = 48, dk: int = 128, dv: int = 128, eps: float = 1e-6) -> gdn_dims:
    return gdn_dims(hk, hv, dk, dv, eps)


def library_path() -> str:
    return _build.LIB


def lib():
    """Load libgdn.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library {path} is missing; build it with "
                                   "`python -m gated_deltanet_linear_pre_gb300.build`")
            L = ctypes.CDLL(path)
            D = ctypes.POINTER(gdn_dims)
            L.gdn_status_string.restype = ctypes.c_char_p
            L.gdn_status_string.argtypes = [ctypes.c_int]
            L.gdn_last_error_string.restype = ctypes.c_char_p
            L.gdn_last_error_string.argtypes = []
            L.gdn_pre.restype = ctypes.c_int
            L.gdn_pre.argtypes = [D, _i32, _i32] + [_p] * 15
            L.gdn_scan_workspace_bytes.restype = _sz
            L.gdn_scan_workspace_bytes.argtypes = [D, _i32, _i32]
            for name in ("gdn_scan", "gdn_scan_fast"):
                getattr(L, name).restype = ctypes.c_int
                getattr(L, name).argtypes = [D, _i32, _i32] + [_p] * 10 + [_sz, _p]
            L.gdn_scan_noalloc.restype = ctypes.c_int
            L.gdn_scan_noalloc.argtypes = [D, _i32, _i32] + [_p] * 9 + [_p]
            L.gdn_scan_noalloc_check.restype = ctypes.c_int
            L.gdn_scan_noalloc_check.argtypes = [_p]
            L.gdn_last_async_error.restype = ctypes.c_int
            L.gdn_last_async_error.argtypes = []
            L.gdn_post.restype = ctypes.c_int
            L.gdn_post.argtypes = [D, _i32, _p, _p, _p, _i32, _p, _p]
            L.gdn_layer_workspace_bytes.restype = _sz
            L.gdn_layer_workspace_bytes.argtypes = [D, _i32, _i32]
            for name in ("gdn_layer", "gdn_layer_fast"):
                getattr(L, name).restype = ctypes.c_int
                getattr(L, name).argtypes = [D, _i32, _i32] + [_p] * 13 + [_i32, _p, _p, _sz, _p]
            L.gdn_scan_check.restype = ctypes.c_int
            L.gdn_scan_check.argtypes = [_p, _p]
            L.gdn_layer_check.restype = ctypes.c_int
            L.gdn_layer_check.argtypes = [D, _i32, _i32, _p, _p]
            L.gdn_scan_selftest_timeout.restype = ctypes.c_int
            L.gdn_scan_selftest_timeout.argtypes = [D, _i32, _i32] + [_p] * 10 + [_sz, _p]
            L.gdn_scan_selftest_one_taker.restype = ctypes.c_int
            L.gdn_scan_selftest_one_taker.argtypes = [D, _i32, _i32] + [_p] * 10 + [_sz, _p]
            L.gdn_scan_selftest_withhold_flag.restype = ctypes.c_int
            L.gdn_scan_selftest_withhold_flag.argtypes = [D, _i32, _i32] + [_p] * 10 + [_sz, _p]
            L.gdn_layer_selftest_stages.restype = ctypes.c_int
            L.gdn_layer_selftest_stages.argtypes = [D, _i32, _i32] + [_p] * 13 + [_i32, _p, _p, _sz, _i32, _i32, _p]
            L.gdn_step.restype = ctypes.c_int
            L.gdn_step.argtypes = [D, _i32] + [_p] * 12 + [_i32, _p, _p]
            _lib = L
    return _lib


def _check(fn: str, status: int):
    if status != 0:
        raise GdnError(fn, status, lib().gdn_last_error_string().decode())


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t, name: str, dtype, shape=None):
    """Device pointer of a contiguous tensor with the documented dtype/shape;
    None passes NULL (allowed only where the ABI allows an empty buffer)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t.data_ptr() if t.numel() else None


def _batch(cu_seqlens, total_tokens):
    if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or cu_seqlens.dim() != 1:
        raise ValueError("cu_seqlens must be a 1-D int32 CUDA tensor")
    return int(cu_seqlens.numel() - 1), int(total_tokens)


def _C(d: gdn_dims) -> int:
    return 2 * d.hk * d.dk + d.hv * d.dv


def gdn_pre(d: gdn_dims, cu_seqlens, total_tokens, qkv, conv_w, hist_in, hist_out, a, b, A_log, dt_bias,
            qn, kn, vc, glog, beta, stream=None):
    n_seq, T = _batch(cu_seqlens, total_tokens)
    C, hk, hv, dk, dv = _C(d), d.hk, d.hv, d.dk, d.dv
    f16, f32 = torch.float16, torch.float32
    st = lib().gdn_pre(ctypes.byref(d), n_seq, T, _ptr(cu_seqlens, "cu_seqlens", torch.int32),
                       _ptr(qkv, "qkv", f16, (T, C)), _ptr(conv_w, "conv_w", f32, (C, 4)),
                       _ptr(hist_in, "hist_in", f16, (n_seq, C, 3)), _ptr(hist_out, "hist_out", f16, (n_seq, C, 3)),
                       _ptr(a, "a", f16, (T, hv)), _ptr(b, "b", f16, (T, hv)),
                       _ptr(A_log, "A_log", f32, (hv,)), _ptr(dt_bias, "dt_bias", f32, (hv,)),
                       _ptr(qn, "qn", f32, (T, hk, dk)), _ptr(kn, "kn", f32, (T, hk, dk)),
                       _ptr(vc, "vc", f32, (T, hv, dv)), _ptr(glog, "glog", f32, (T, hv)),
                       _ptr(beta, "beta", f32, (T, hv)), _stream(stream))
    _check("gdn_pre", st)


def gdn_scan_workspace_bytes(d: gdn_dims, n_seq: int, total_tokens: int) -> int:
    return int(lib().gdn_scan_workspace_bytes(ctypes.byref(d), n_seq, total_tokens))


def gdn_scan(d: gdn_dims, cu_seqlens, total_tokens, qn, kn, vc, glog, beta, S_in, S_out, o,
             workspace=None, stream=None):
    _scan("gdn_scan", d, cu_seqlens, total_tokens, qn, kn, vc, glog, beta, S_in, S_out, o, workspace, stream)


def gdn_scan_fast(d: gdn_dims, cu_seqlens, total_tokens, qn, kn, vc, glog, beta, S_in, S_out, o,
                  workspace=None, stream=None):
    """gdn_scan with one-pass bf16 tensor-core products (faster, less accurate)."""
    _scan("gdn_scan_fast", d, cu_seqlens, total_tokens, qn, kn, vc, glog, beta, S_in, S_out, o, workspace, stream)


def _scan(name, d, cu_seqlens, total_tokens, qn, kn, vc, glog, beta, S_in, S_out, o, workspace, stream):
    n_seq, T = _batch(cu_seqlens, total_tokens)
    hk, hv, dk, dv = d.hk, d.hv, d.dk, d.dv
    f32 = torch.float32
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _ptr(workspace, "workspace", torch.uint8), workspace.numel()
    st = getattr(lib(), name)(ctypes.byref(d), n_seq, T, _ptr(cu_seqlens, "cu_seqlens", torch.int32),
                        _ptr(qn, "qn", f32, (T, hk, dk)), _ptr(kn, "kn", f32, (T, hk, dk)),
                        _ptr(vc, "vc", f32, (T, hv, dv)), _ptr(glog, "glog", f32, (T, hv)),
                        _ptr(beta, "beta", f32, (T, hv)), _ptr(S_in, "S_in", f32, (n_seq, hv, dk, dv)),
                        _ptr(S_out, "S_out", f32, (n_seq, hv, dk, dv)), _ptr(o, "o", f32, (T, hv, dv)),
                        ws_ptr, ws_bytes, _stream(stream))
    _check(name, st)


def gdn_scan_noalloc(d: gdn_dims, cu_seqlens, total_tokens, qn, kn, vc, glog, beta, S_in, S_out, o, stream=None):
    """gdn_scan with the library's own fixed scratch instead of a workspace, for
    callers that cannot allocate device memory (see include/gdn.h)."""
    n_seq, T = _batch(cu_seqlens, total_tokens)
    hk, hv, dk, dv = d.hk, d.hv, d.dk, d.dv
    f32 = torch.float32
    st = lib().gdn_scan_noalloc(ctypes.byref(d), n_seq, T, _ptr(cu_seqlens, "cu_seqlens", torch.int32),
                                _ptr(qn, "qn", f32, (T, hk, dk)), _ptr(kn, "kn", f32, (T, hk, dk)),
                                _ptr(vc, "vc", f32, (T, hv, dv)), _ptr(glog, "glog", f32, (T, hv)),
                                _ptr(beta, "beta", f32, (T, hv)), _ptr(S_in, "S_in", f32, (n_seq, hv, dk, dv)),
                                _ptr(S_out, "S_out", f32, (n_seq, hv, dk, dv)), _ptr(o, "o", f32, (T, hv, dv)),
                                _stream(stream))
    _check("gdn_scan_noalloc", st)


def gdn_post(d: gdn_dims, total_tokens, o, z, gamma, out_f32: bool, y, stream=None):
    T, hv, dv = int(total_tokens), d.hv, d.dv
    ydt = torch.float32 if out_f32 else torch.float16
    st = lib().gdn_post(ctypes.byref(d), T, _ptr(o, "o", torch.float32, (T, hv, dv)),
                        _ptr(z, "z", torch.float16, (T, hv, dv)), _ptr(gamma, "gamma", torch.float32, (dv,)),
                        1 if out_f32 else 0, _ptr(y, "y", ydt, (T, hv, dv)), _stream(stream))
    _check("gdn_post", st)


def gdn_layer_workspace_bytes(d: gdn_dims, n_seq: int, total_tokens: int) -> int:
    return int(lib().gdn_layer_workspace_bytes(ctypes.byref(d), n_seq, total_tokens))


def gdn_layer(d: gdn_dims, cu_seqlens, total_tokens, qkv, conv_w, hist_in, hist_out, a, b, z, A_log, dt_bias,
              gamma, S_in, S_out, out_f32: bool, y, workspace, stream=None):
    _layer("gdn_layer", d, cu_seqlens, total_tokens, qkv, conv_w, hist_in, hist_out, a, b, z, A_log, dt_bias,
           gamma, S_in, S_out, out_f32, y, workspace, stream)


def gdn_layer_fast(d: gdn_dims, cu_seqlens, total_tokens, qkv, conv_w, hist_in, hist_out, a, b, z, A_log,
                   dt_bias, gamma, S_in, S_out, out_f32: bool, y, workspace, stream=None):
    """gdn_layer with one-pass bf16 tensor-core products in the scan (faster, less accurate)."""
    _layer("gdn_layer_fast", d, cu_seqlens, total_tokens, qkv, conv_w, hist_in, hist_out, a, b, z, A_log, dt_bias,
           gamma, S_in, S_out, out_f32, y, workspace, stream)


def gdn_layer_selftest_stages(d: gdn_dims, cu_seqlens, total_tokens, qkv, conv_w, hist_in, hist_out, a, b, z,
                              A_log, dt_bias, gamma, S_in, S_out, out_f32: bool, y, workspace, fast: bool,
                              stages: int, stream=None):
    """Test and timing hook: only the gdn_layer stages in the mask `stages` (1 pre, 2 scan, 4 post)."""
    _layer("gdn_layer_selftest_stages", d, cu_seqlens, total_tokens, qkv, conv_w, hist_in, hist_out, a, b, z, A_log,
           dt_bias, gamma, S_in, S_out, out_f32, y, workspace, stream, extra=(1 if fast else 0, int(stages)))


def _layer(name, d, cu_seqlens, total_tokens, qkv, conv_w, hist_in, hist_out, a, b, z, A_log, dt_bias,
           gamma, S_in, S_out, out_f32, y, workspace, stream, extra=()):
    n_seq, T = _batch(cu_seqlens, total_tokens)
    C, hv, dk, dv = _C(d), d.hv, d.dk, d.dv
    f16, f32 = torch.float16, torch.float32
    ydt = f32 if out_f32 else f16
    st = getattr(lib(), name)(ctypes.byref(d), n_seq, T, _ptr(cu_seqlens, "cu_seqlens", torch.int32),
                         _ptr(qkv, "qkv", f16, (T, C)), _ptr(conv_w, "conv_w", f32, (C, 4)),
                         _ptr(hist_in, "hist_in", f16, (n_seq, C, 3)),
                         _ptr(hist_out, "hist_out", f16, (n_seq, C, 3)),
                         _ptr(a, "a", f16, (T, hv)), _ptr(b, "b", f16, (T, hv)), _ptr(z, "z", f16, (T, hv, dv)),
                         _ptr(A_log, "A_log", f32, (hv,)), _ptr(dt_bias, "dt_bias", f32, (hv,)),
                         _ptr(gamma, "gamma", f32, (dv,)), _ptr(S_in, "S_in", f32, (n_seq, hv, dk, dv)),
                         _ptr(S_out, "S_out", f32, (n_seq, hv, dk, dv)), 1 if out_f32 else 0,
                         _ptr(y, "y", ydt, (T, hv, dv)), _ptr(workspace, "workspace", torch.uint8),
                         workspace.numel() if workspace is not None else 0, *extra, _stream(stream))
    _check(name, st)


def gdn_step(d: gdn_dims, n_seq: int, qkv, conv_w, hist_in, hist_out, a, b, z, A_log, dt_bias, gamma, S_in, S_out,
             out_f32: bool, y, stream=None):
    """One decode step: one token per sequence (qkv [n_seq, C]) through pre, the recurrence and post."""
    n = int(n_seq)
    C, hv, dk, dv = _C(d), d.hv, d.dk, d.dv
    f16, f32 = torch.float16, torch.float32
    ydt = f32 if out_f32 else f16
    st = lib().gdn_step(ctypes.byref(d), n, _ptr(qkv, "qkv", f16, (n, C)), _ptr(conv_w, "conv_w", f32, (C, 4)),
                        _ptr(hist_in, "hist_in", f16, (n, C, 3)), _ptr(hist_out, "hist_out", f16, (n, C, 3)),
                        _ptr(a, "a", f16, (n, hv)), _ptr(b, "b", f16, (n, hv)), _ptr(z, "z", f16, (n, hv, dv)),
                        _ptr(A_log, "A_log", f32, (hv,)), _ptr(dt_bias, "dt_bias", f32, (hv,)),
                        _ptr(gamma, "gamma", f32, (dv,)), _ptr(S_in, "S_in", f32, (n, hv, dk, dv)),
                        _ptr(S_out, "S_out", f32, (n, hv, dk, dv)), 1 if out_f32 else 0,
                        _ptr(y, "y", ydt, (n, hv, dv)), _stream(stream))
    _check("gdn_step", st)


def gdn_scan_check(workspace, stream=None):
    """Raise GdnError (GDN_ERR_TIMEOUT) if the last scan on this workspace reported an expired wait;
    synchronises the stream."""
    _check("gdn_scan_check", lib().gdn_scan_check(_ptr(workspace, "workspace", torch.uint8), _stream(stream)))


def gdn_scan_noalloc_check(stream=None):
    """As gdn_scan_check for the last gdn_scan_noalloc on the current device; synchronises the stream."""
    _check("gdn_scan_noalloc_check", lib().gdn_scan_noalloc_check(_stream(stream)))


def gdn_last_async_error():
    """Raise GdnError (GDN_ERR_CUDA) if the library has seen a fault that left the CUDA context
    unusable; never synchronises."""
    _check("gdn_last_async_error", lib().gdn_last_async_error())


def gdn_layer_check(d: gdn_dims, n_seq: int, total_tokens: int, workspace, stream=None):
    """As gdn_scan_check for a gdn_layer workspace."""
    _check("gdn_layer_check", lib().gdn_layer_check(ctypes.byref(d), int(n_seq), int(total_tokens),
                                                    _ptr(workspace, "workspace", torch.uint8), _stream(stream)))


def gdn_scan_selftest_timeout(d: gdn_dims, cu_seqlens, total_tokens, qn, kn, vc, glog, beta, S_in, S_out, o,
                              workspace, stream=None):
    """Test hook of the failure report: gdn_scan with one operand copy withheld (outputs invalid)."""
    n_seq, T = _batch(cu_seqlens, total_tokens)
    hk, hv, dk, dv = d.hk, d.hv, d.dk, d.dv
    f32 = torch.float32
    st = lib().gdn_scan_selftest_timeout(
        ctypes.byref(d), n_seq, T, _ptr(cu_seqlens, "cu_seqlens", torch.int32), _ptr(qn, "qn", f32, (T, hk, dk)),
        _ptr(kn, "kn", f32, (T, hk, dk)), _ptr(vc, "vc", f32, (T, hv, dv)), _ptr(glog, "glog", f32, (T, hv)),
        _ptr(beta, "beta", f32, (T, hv)), _ptr(S_in, "S_in", f32, (n_seq, hv, dk, dv)),
        _ptr(S_out, "S_out", f32, (n_seq, hv, dk, dv)), _ptr(o, "o", f32, (T, hv, dv)),
        _ptr(workspace, "workspace", torch.uint8), workspace.numel() if workspace is not None else 0,
        _stream(stream))
    _check("gdn_scan_selftest_timeout", st)


def gdn_scan_selftest_one_taker(d: gdn_dims, cu_seqlens, total_tokens, qn, kn, vc, glog, beta, S_in, S_out, o,
                                workspace, stream=None):
    """Test hook of prep's progress guarantee: gdn_scan with no SM kept for prep after its first round."""
    n_seq, T = _batch(cu_seqlens, total_tokens)
    hk, hv, dk, dv = d.hk, d.hv, d.dk, d.dv
    f32 = torch.float32
    st = lib().gdn_scan_selftest_one_taker(
        ctypes.byref(d), n_seq, T, _ptr(cu_seqlens, "cu_seqlens", torch.int32), _ptr(qn, "qn", f32, (T, hk, dk)),
        _ptr(kn, "kn", f32, (T, hk, dk)), _ptr(vc, "vc", f32, (T, hv, dv)), _ptr(glog, "glog", f32, (T, hv)),
        _ptr(beta, "beta", f32, (T, hv)), _ptr(S_in, "S_in", f32, (n_seq, hv, dk, dv)),
        _ptr(S_out, "S_out", f32, (n_seq, hv, dk, dv)), _ptr(o, "o", f32, (T, hv, dv)),
        _ptr(workspace, "workspace", torch.uint8), workspace.numel() if workspace is not None else 0,
        _stream(stream))
    _check("gdn_scan_selftest_one_taker", st)


def gdn_scan_selftest_withhold_flag(d: gdn_dims, cu_seqlens, total_tokens, qn, kn, vc, glog, beta, S_in, S_out, o,
                                    workspace, stream=None):
    """Test hook of the wait across kernels: gdn_scan with one prep ready flag left unset (outputs invalid)."""
    n_seq, T = _batch(cu_seqlens, total_tokens)
    hk, hv, dk, dv = d.hk, d.hv, d.dk, d.dv
    f32 = torch.float32
    st = lib().gdn_scan_selftest_withhold_flag(
        ctypes.byref(d), n_seq, T, _ptr(cu_seqlens, "cu_seqlens", torch.int32), _ptr(qn, "qn", f32, (T, hk, dk)),
        _ptr(kn, "kn", f32, (T, hk, dk)), _ptr(vc, "vc", f32, (T, hv, dv)), _ptr(glog, "glog", f32, (T, hv)),
        _ptr(beta, "beta", f32, (T, hv)), _ptr(S_in, "S_in", f32, (n_seq, hv, dk, dv)),
        _ptr(S_out, "S_out", f32, (n_seq, hv, dk, dv)), _ptr(o, "o", f32, (T, hv, dv)),
        _ptr(workspace, "workspace", torch.uint8), workspace.numel() if workspace is not None else 0,
        _stream(stream))
    _check("gdn_scan_selftest_withhold_flag", st)
