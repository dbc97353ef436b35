"""GB300 (sm_103a) scaled dot-product attention forward pass.

Python binding of the C ABI in include/sdpa.h.  Every step of the computation
runs in the CUDA library; these functions only marshal PyTorch CUDA tensors
(used for device memory and streams) into the C call.
"""
from __future__ import annotations

import ctypes
import math

import torch

from . import _abi
from ._abi import SdpaError, check, lib, status_string

__all__ = ["sdpa_fwd", "sdpa_fwd_fp8", "sdpa_fwd_ex", "sdpa_fwd_fp8_ex", "sdpa_fwd_decode", "sdpa_fwd_decode_noalloc",
           "sdpa_bwd", "bwd_workspace_bytes", "sdpa_bwd_fp8", "bwd_fp8_workspace_bytes",
           "decode_workspace_bytes", "sdpa_status_string", "sdpa_device_error", "SdpaError", "lib"]

_DTYPE = {torch.bfloat16: _abi.SDPA_DTYPE_BF16, torch.float16: _abi.SDPA_DTYPE_FP16}


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_ptr(stream, device_index: int):
    """cudaStream_t for the call: the given stream, else the current stream
    of the tensors' device (read without building a Stream object)."""
    if stream is None:
        if _raw_stream is not None:
            return ctypes.c_void_p(_raw_stream(device_index))
        stream = torch.cuda.current_stream(device_index)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _run(device_index: int, fn, *args) -> None:
    """Call ``fn`` with the tensors' device current: the C library works on
    the current CUDA device (its SM count, kernel attributes and the decode
    scratch are per device), so a call on tensors of another device switches
    to it for the duration of the call."""
    if torch.cuda.current_device() != device_index:
        with torch.cuda.device(device_index):
            check(fn(*args))
    else:
        check(fn(*args))


def _shapes(q, k, v):
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("Q, K, V must be [B, S, H, D]")
    B, Sq, Hq, D = q.shape
    _, Skv, Hkv, _ = k.shape
    return B, Hq, Hkv, Sq, Skv, D


def sdpa_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor | None = None, *,
             causal: bool = False, scale: float | None = None, stream=None) -> torch.Tensor:
    """O = softmax(Q K^T * scale [+ causal mask]) V on the GPU.

    q: [B, Sq, Hq, D], k and v: [B, Skv, Hkv, D], bf16 or fp16 contiguous CUDA
    tensors (shape agreement is checked by the library).  Returns ``o``
    (allocated like ``q`` when not given)."""
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("inputs must be contiguous CUDA tensors")
    if k.shape != v.shape or k.shape[0] != q.shape[0] or k.shape[3] != q.shape[3] or q.dtype != k.dtype \
            or q.dtype != v.dtype:
        raise ValueError("K and V must be [B, Skv, Hkv, D] like Q, with Q's dtype")
    B, Hq, Hkv, Sq, Skv, D = _shapes(q, k, v)
    if o is None:
        o = torch.empty_like(q)
    elif not o.is_cuda or not o.is_contiguous() or o.shape != q.shape or o.dtype != q.dtype:
        raise ValueError("o must be a contiguous CUDA tensor shaped and typed like q")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dt = _DTYPE.get(q.dtype, 99)
    _run(q.device.index, lib().sdpa_fwd, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, Hq, Hkv, Sq, Skv, D,
                         float(scale), int(bool(causal)), dt, _stream_ptr(stream, q.device.index))
    return o


def sdpa_fwd_fp8(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor | None = None, *,
                 descale_q: float, descale_k: float, descale_v: float, causal: bool = False,
                 scale: float | None = None, stream=None) -> torch.Tensor:
    """FP8 E4M3 inputs (``torch.float8_e4m3fn`` or uint8 codes) with
    per-tensor descales; bf16 output."""
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous() or t.element_size() != 1:
            raise ValueError("inputs must be contiguous 1-byte CUDA tensors")
    B, Hq, Hkv, Sq, Skv, D = _shapes(q, k, v)
    if o is None:
        o = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    elif not o.is_cuda or not o.is_contiguous() or o.shape != q.shape or o.dtype != torch.bfloat16:
        raise ValueError("o must be a contiguous bf16 CUDA tensor shaped like q")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    _run(q.device.index, lib().sdpa_fwd_fp8, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, Hq, Hkv, Sq, Skv, D,
                             float(scale), float(descale_q), float(descale_k), float(descale_v),
                             int(bool(causal)), _stream_ptr(stream, q.device.index))
    return o


def _layout(t: torch.Tensor) -> _abi.Layout:
    """Strides of a [B, S, H, D] tensor view (D contiguous) as sdpa_layout_t."""
    if t.dim() != 4 or t.stride(3) != 1:
        raise ValueError("tensors must be 4-D [B, S, H, D] views with a contiguous last dimension")
    return _abi.Layout(t.stride(0), t.stride(1), t.stride(2))


def _lse_ptr(lse, B, Hq, Sq):
    if lse is None:
        return None
    if not lse.is_cuda or lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != (B, Hq, Sq):
        raise ValueError("lse must be a contiguous float32 CUDA tensor [B, Hq, Sq]")
    return lse.data_ptr()


def sdpa_fwd_ex(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, lse: torch.Tensor | None = None,
                *, causal: bool = False, scale: float | None = None, stream=None) -> torch.Tensor:
    """sdpa_fwd on [B, S, H, D] views with any strides the library accepts
    (e.g. a BHSD tensor permuted to [B, S, H, D]), writing O through ``o``'s
    strides and, when ``lse`` ([B, Hq, Sq] float32) is given, the log-sum-exp
    of every row's scores.  Returns ``o``."""
    for t in (q, k, v, o):
        if not t.is_cuda:
            raise ValueError("tensors must be CUDA tensors")
    if q.dtype != k.dtype or q.dtype != v.dtype or o.dtype != q.dtype or tuple(o.shape) != tuple(q.shape):
        raise ValueError("q, k, v, o must share a dtype; o is shaped like q")
    B, Hq, Hkv, Sq, Skv, D = _shapes(q, k, v)
    if tuple(k.shape) != tuple(v.shape):
        raise ValueError("K and V must have the same shape")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    lq, lk, lv, lo = _layout(q), _layout(k), _layout(v), _layout(o)
    _run(q.device.index, lib().sdpa_fwd_ex, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), _lse_ptr(lse, B, Hq, Sq),
                            B, Hq, Hkv, Sq, Skv, D, ctypes.byref(lq), ctypes.byref(lk), ctypes.byref(lv),
                            ctypes.byref(lo), float(scale), int(bool(causal)), _DTYPE.get(q.dtype, 99),
                            _stream_ptr(stream, q.device.index))
    return o


def sdpa_fwd_fp8_ex(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                    lse: torch.Tensor | None = None, *, descale_q: float, descale_k: float, descale_v: float,
                    causal: bool = False, scale: float | None = None, stream=None) -> torch.Tensor:
    """sdpa_fwd_fp8 with strided views and an optional LSE, as sdpa_fwd_ex."""
    for t in (q, k, v):
        if not t.is_cuda or t.element_size() != 1:
            raise ValueError("inputs must be 1-byte CUDA tensors")
    if not o.is_cuda or o.dtype != torch.bfloat16 or tuple(o.shape) != tuple(q.shape):
        raise ValueError("o must be a bf16 CUDA tensor shaped like q")
    B, Hq, Hkv, Sq, Skv, D = _shapes(q, k, v)
    if tuple(k.shape) != tuple(v.shape):
        raise ValueError("K and V must have the same shape")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    lq, lk, lv, lo = _layout(q), _layout(k), _layout(v), _layout(o)
    _run(q.device.index, lib().sdpa_fwd_fp8_ex, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), _lse_ptr(lse, B, Hq, Sq),
                                B, Hq, Hkv, Sq, Skv, D, ctypes.byref(lq), ctypes.byref(lk), ctypes.byref(lv),
                                ctypes.byref(lo), float(scale), float(descale_q), float(descale_k),
                                float(descale_v), int(bool(causal)), _stream_ptr(stream, q.device.index))
    return o


def decode_workspace_bytes(B: int, Hq: int, Hkv: int, Sq: int, Skv: int, D: int) -> int:
    """Workspace bytes sdpa_fwd_decode needs for this shape on the current
    device (0: the pass is not split)."""
    return int(lib().sdpa_decode_workspace_bytes(B, Hq, Hkv, Sq, Skv, D))


def sdpa_fwd_decode(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                    lse: torch.Tensor | None = None, *, workspace: torch.Tensor | None = None,
                    scale: float | None = None, stream=None) -> torch.Tensor:
    """Non-causal decode-shaped pass (few query rows, long K/V): the query
    heads of each KV head are stacked into one tile, and with ``workspace``
    (a CUDA tensor of at least :func:`decode_workspace_bytes` bytes) the key
    sequence is split across the GPU.  Strided views and ``lse`` as for
    :func:`sdpa_fwd_ex`.  Returns ``o``."""
    for t in (q, k, v, o):
        if not t.is_cuda:
            raise ValueError("tensors must be CUDA tensors")
    if q.dtype != k.dtype or q.dtype != v.dtype or o.dtype != q.dtype or tuple(o.shape) != tuple(q.shape):
        raise ValueError("q, k, v, o must share a dtype; o is shaped like q")
    B, Hq, Hkv, Sq, Skv, D = _shapes(q, k, v)
    if tuple(k.shape) != tuple(v.shape):
        raise ValueError("K and V must have the same shape")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    ws, ws_bytes = None, 0
    if workspace is not None:
        if not workspace.is_cuda or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    lq, lk, lv, lo = _layout(q), _layout(k), _layout(v), _layout(o)
    _run(q.device.index, lib().sdpa_fwd_decode, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), _lse_ptr(lse, B, Hq, Sq),
                                B, Hq, Hkv, Sq, Skv, D, ctypes.byref(lq), ctypes.byref(lk), ctypes.byref(lv),
                                ctypes.byref(lo), float(scale), _DTYPE.get(q.dtype, 99), ws, ws_bytes,
                                _stream_ptr(stream, q.device.index))
    return o


def sdpa_fwd_decode_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                            lse: torch.Tensor | None = None, *, scale: float | None = None,
                            stream=None) -> torch.Tensor:
    """:func:`sdpa_fwd_decode` with the library's own device scratch instead
    of a workspace (allocates nothing; calls must not run concurrently)."""
    for t in (q, k, v, o):
        if not t.is_cuda:
            raise ValueError("tensors must be CUDA tensors")
    if q.dtype != k.dtype or q.dtype != v.dtype or o.dtype != q.dtype or tuple(o.shape) != tuple(q.shape):
        raise ValueError("q, k, v, o must share a dtype; o is shaped like q")
    B, Hq, Hkv, Sq, Skv, D = _shapes(q, k, v)
    if tuple(k.shape) != tuple(v.shape):
        raise ValueError("K and V must have the same shape")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    lq, lk, lv, lo = _layout(q), _layout(k), _layout(v), _layout(o)
    _run(q.device.index, lib().sdpa_fwd_decode_noalloc, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                        _lse_ptr(lse, B, Hq, Sq), B, Hq, Hkv, Sq, Skv, D, ctypes.byref(lq),
                                        ctypes.byref(lk), ctypes.byref(lv), ctypes.byref(lo), float(scale),
                                        _DTYPE.get(q.dtype, 99), _stream_ptr(stream, q.device.index))
    return o


def bwd_workspace_bytes(B: int, Hq: int, Sq: int, D: int) -> int:
    """Workspace bytes :func:`sdpa_bwd` needs."""
    return int(lib().sdpa_bwd_workspace_bytes(B, Hq, Sq, D))


def sdpa_bwd(q, k, v, o, do, lse, dq=None, dk=None, dv=None, *, causal: bool = False, scale: float | None = None,
             workspace=None, stream=None):
    """Gradients (dq, dk, dv) of sum(do * o) for o = sdpa_fwd(q, k, v) on
    contiguous [B, S, H, D] bf16 / fp16 CUDA tensors; ``lse`` is the
    forward's [B, Hq, Sq] float32 log-sum-exp (from :func:`sdpa_fwd_ex`).
    Outputs and the workspace are allocated when not given."""
    for t in (q, k, v, o, do):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != q.dtype:
            raise ValueError("q, k, v, o, do must be contiguous CUDA tensors of one dtype")
    B, Hq, Hkv, Sq, Skv, D = _shapes(q, k, v)
    if tuple(o.shape) != tuple(q.shape) or tuple(do.shape) != tuple(q.shape) or tuple(k.shape) != tuple(v.shape):
        raise ValueError("o and do must be shaped like q, v like k")
    lse_ptr = _lse_ptr(lse, B, Hq, Sq)
    if lse_ptr is None:
        raise ValueError("the forward's lse is required")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t, like in ((dq, q), (dk, k), (dv, v)):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != like.dtype or t.shape != like.shape:
            raise ValueError("gradients must be contiguous CUDA tensors shaped and typed like their inputs")
    if workspace is None:
        workspace = torch.empty(bwd_workspace_bytes(B, Hq, Sq, D), dtype=torch.uint8, device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    _run(q.device.index, lib().sdpa_bwd, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse_ptr,
                         dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, Sq, Skv, D, float(scale),
                         int(bool(causal)), _DTYPE.get(q.dtype, 99), workspace.data_ptr(),
                         workspace.numel() * workspace.element_size(), _stream_ptr(stream, q.device.index))
    return dq, dk, dv


def bwd_fp8_workspace_bytes(B: int, Hq: int, Sq: int, D: int) -> int:
    """Workspace bytes :func:`sdpa_bwd_fp8` needs."""
    return int(lib().sdpa_bwd_fp8_workspace_bytes(B, Hq, Sq, D))


def sdpa_bwd_fp8(q8, k8, v8, o, do8, lse, dq=None, dk=None, dv=None, *, descale_q: float, descale_k: float,
                 descale_v: float, descale_do: float, scale_ds: float, amax_ds=None, causal: bool = False,
                 scale: float | None = None, workspace=None, stream=None):
    """FP8 backward pass: gradients (dq, dk, dv), bf16, of sum(do * o) for
    o = sdpa_fwd_fp8(q8, k8, v8).  ``q8``, ``k8``, ``v8`` are E4M3 and ``do8``
    E5M2 (``torch.float8_e4m3fn`` / ``torch.float8_e5m2`` or uint8 codes),
    contiguous [B, S, H, D] CUDA tensors with per-tensor descales; ``o`` is
    the forward's bf16 output and ``lse`` its [B, Hq, Sq] float32
    log-sum-exp.  ``scale_ds`` scales dS before its E5M2 rounding; if
    ``amax_ds`` (a 1-element float32 CUDA tensor) is given it receives
    max |dS| of this call.  Outputs and the workspace are allocated when not
    given."""
    for t in (q8, k8, v8, do8):
        if not t.is_cuda or not t.is_contiguous() or t.element_size() != 1:
            raise ValueError("q8, k8, v8, do8 must be contiguous 1-byte CUDA tensors")
    B, Hq, Hkv, Sq, Skv, D = _shapes(q8, k8, v8)
    if tuple(do8.shape) != tuple(q8.shape) or tuple(o.shape) != tuple(q8.shape) or tuple(k8.shape) != tuple(v8.shape):
        raise ValueError("o and do8 must be shaped like q8, v8 like k8")
    if not o.is_cuda or not o.is_contiguous() or o.dtype != torch.bfloat16:
        raise ValueError("o must be a contiguous bf16 CUDA tensor")
    lse_ptr = _lse_ptr(lse, B, Hq, Sq)
    if lse_ptr is None:
        raise ValueError("the forward's lse is required")
    dq = torch.empty(q8.shape, dtype=torch.bfloat16, device=q8.device) if dq is None else dq
    dk = torch.empty(k8.shape, dtype=torch.bfloat16, device=q8.device) if dk is None else dk
    dv = torch.empty(v8.shape, dtype=torch.bfloat16, device=q8.device) if dv is None else dv
    for t, like in ((dq, q8), (dk, k8), (dv, v8)):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != torch.bfloat16 or t.shape != like.shape:
            raise ValueError("gradients must be contiguous bf16 CUDA tensors shaped like their inputs")
    amax_ptr = None
    if amax_ds is not None:
        if not amax_ds.is_cuda or amax_ds.dtype != torch.float32 or amax_ds.numel() < 1:
            raise ValueError("amax_ds must be a float32 CUDA tensor")
        amax_ptr = amax_ds.data_ptr()
    if workspace is None:
        workspace = torch.empty(bwd_fp8_workspace_bytes(B, Hq, Sq, D), dtype=torch.uint8, device=q8.device)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    _run(q8.device.index, lib().sdpa_bwd_fp8, q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), o.data_ptr(), do8.data_ptr(), lse_ptr,
                             dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, Sq, Skv, D, float(scale),
                             int(bool(causal)), float(descale_q), float(descale_k), float(descale_v),
                             float(descale_do), float(scale_ds), amax_ptr, workspace.data_ptr(),
                             workspace.numel() * workspace.element_size(), _stream_ptr(stream, q8.device.index))
    return dq, dk, dv


def sdpa_status_string(status: int) -> str:
    return status_string(status)


def sdpa_device_error() -> int:
    """Read and clear the device error word (synchronises the device)."""
    code = ctypes.c_uint(0)
    check(lib().sdpa_device_error(ctypes.byref(code)))
    return int(code.value)
