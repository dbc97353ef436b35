"""fp64 CPU oracle for the scaled dot-product attention forward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product package never imports it, and the oracle imports nothing from the
product package: the two share no code.

The arithmetic lives in ``sdpa_oracle.c`` (a plain C loop nest, built with gcc
and OpenMP over query rows).  This module only builds that library and marshals
arrays into it.  What it computes is the definition in the codelab "Attention
on GPU (cuDNN and TransformerEngine)", section 1 ("How attention works") and
section 4 ("Implement attention from scratch"):

    O = softmax(Q K^T * scale [+ causal mask]) V

with the causal mask of section 7 (query row i sees keys 0..i) and the grouped
KV heads of section 9 (query head hq reads KV head hq // (Hq // Hkv)).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sdpa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

DTYPES = {"bf16": 0, "fp16": 1, "e4m3": 2, "f32": 3, "f64": 4}
_ELEM_BYTES = {"bf16": 2, "fp16": 2, "e4m3": 1, "f32": 4, "f64": 8}

_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the C oracle into a shared library (gcc, -O2, OpenMP)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall",
           "-Wextra", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(lib):
    cvp, cl, ci, cd = ctypes.c_void_p, ctypes.c_long, ctypes.c_int, ctypes.c_double
    lib.oracle_sdpa_rows.restype = ci
    lib.oracle_sdpa_rows.argtypes = [cvp, cvp, cvp, ci, cd, cd, cd, cl, cl, cl, cl, cl, cl,
                                     cd, ci, cvp, cl, cvp, cvp, cvp, ci]
    lib.oracle_sdpa_fwd.restype = ci
    lib.oracle_sdpa_fwd.argtypes = [cvp, cvp, cvp, ci, cd, cd, cd, cl, cl, cl, cl, cl, cl,
                                    cd, ci, cvp, cvp, ci]
    lib.oracle_sdpa_bwd.restype = ci
    lib.oracle_sdpa_bwd.argtypes = [cvp, cvp, cvp, cvp, ci, cl, cl, cl, cl, cl, cl, cd, ci, cvp, cvp, cvp, ci]
    lib.oracle_decode.restype = cd
    lib.oracle_decode.argtypes = [cvp, cl, ci, cd]
    lib.oracle_max_threads.restype = ci
    lib.oracle_max_threads.argtypes = []
    return lib


def load_library(path: str | None = None):
    """Load (building first if needed) the oracle library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def _raw(x, dtype: str) -> np.ndarray:
    """Contiguous numpy view of the raw element codes of ``x``.

    ``x`` is a numpy array or a CPU torch tensor.  bf16 / fp16 / e4m3 tensors
    are reinterpreted as their integer codes (no value conversion happens
    here; the C library decodes the codes itself)."""
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(x, torch.Tensor):
        x = x.detach().contiguous().cpu()
        if dtype in ("bf16", "fp16"):
            x = x.view(torch.int16)
        elif dtype == "e4m3":
            x = x.view(torch.uint8)
        x = x.numpy()
    a = np.ascontiguousarray(x)
    if a.dtype.itemsize != _ELEM_BYTES[dtype]:
        raise TypeError(f"array of itemsize {a.dtype.itemsize} does not hold {dtype} codes")
    return a


def _check_shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("Q, K, V must be 4-D [B, S, H, D]")
    B, Sq, Hq, D = q.shape
    Bk, Skv, Hkv, Dk = k.shape
    if k.shape != v.shape or Bk != B or Dk != D:
        raise ValueError(f"incompatible shapes {q.shape} {k.shape} {v.shape}")
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    return B, Hq, Hkv, Sq, Skv, D


def sdpa_reference(q, k, v, *, causal: bool, scale: float | None = None, dtype: str = "bf16",
                   descales=(1.0, 1.0, 1.0), rows=None, threads: int = 0,
                   return_weights: bool = False, return_lse: bool = False, lib=None):
    """fp64 attention output.

    q: [B, Sq, Hq, D]; k, v: [B, Skv, Hkv, D] (numpy or CPU torch), holding
    ``dtype`` elements ("bf16", "fp16", "e4m3", "f32" or "f64").  For "e4m3"
    the decoded codes are multiplied by the per-tensor ``descales``.
    ``scale`` defaults to 1/sqrt(D) (section 4 of the codelab).

    Returns float64 [B, Sq, Hq, D], or, when ``rows`` (flat indices
    (b*Sq + i)*Hq + hq) is given, float64 [len(rows), D].  With
    ``return_weights`` (rows required) also returns the [len(rows), Skv]
    softmax weights.  With ``return_lse`` also returns the log-sum-exp of each
    row's visible scores, log(sum_j exp(s_j)) -- the log of the softmax
    denominator of section 1 -- as float64 [B, Hq, Sq] (whole pass) or
    [len(rows)] (rows); with both flags the order is (out, weights, lse).
    :func:`last_threads` reports how many threads the call used.
    """
    lib = lib or load_library()
    qa, ka, va = _raw(q, dtype), _raw(k, dtype), _raw(v, dtype)
    B, Hq, Hkv, Sq, Skv, D = _check_shapes(qa, ka, va)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    code = DTYPES[dtype]
    dq, dk, dv = (float(s) for s in descales)
    global _last_threads
    if rows is None:
        if return_weights:
            raise ValueError("return_weights needs explicit rows")
        out = np.empty((B, Sq, Hq, D), dtype=np.float64)
        lse = np.empty((B, Hq, Sq), dtype=np.float64) if return_lse else None
        nt = lib.oracle_sdpa_fwd(qa.ctypes.data, ka.ctypes.data, va.ctypes.data, code, dq, dk, dv,
                                 B, Hq, Hkv, Sq, Skv, D, float(scale), int(bool(causal)),
                                 out.ctypes.data, lse.ctypes.data if lse is not None else None, int(threads))
        if nt < 0:
            raise ValueError("oracle rejected the arguments")
        _last_threads = nt
        return (out, lse) if return_lse else out
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.empty((r.size, D), dtype=np.float64)
    w = np.empty((r.size, Skv), dtype=np.float64) if return_weights else None
    lse = np.empty((r.size,), dtype=np.float64) if return_lse else None
    nt = lib.oracle_sdpa_rows(qa.ctypes.data, ka.ctypes.data, va.ctypes.data, code, dq, dk, dv,
                              B, Hq, Hkv, Sq, Skv, D, float(scale), int(bool(causal)),
                              r.ctypes.data, r.size, out.ctypes.data,
                              w.ctypes.data if w is not None else None,
                              lse.ctypes.data if lse is not None else None, int(threads))
    if nt < 0:
        raise ValueError("oracle rejected the arguments")
    _last_threads = nt
    res = (out,) + ((w,) if return_weights else ()) + ((lse,) if return_lse else ())
    return res[0] if len(res) == 1 else res


_last_threads = 0


def sdpa_backward_reference(q, k, v, do, *, causal: bool, scale: float | None = None, dtype: str = "bf16",
                            threads: int = 0, lib=None):
    """fp64 gradients (dQ, dK, dV) of sum(dO * O) for O = attention(Q, K, V):
    dQ [B, Sq, Hq, D], dK and dV [B, Skv, Hkv, D] (float64).  ``do`` has Q's
    shape and element type ("bf16", "fp16", "f32" or "f64")."""
    global _last_threads
    lib = lib or load_library()
    qa, ka, va, da = _raw(q, dtype), _raw(k, dtype), _raw(v, dtype), _raw(do, dtype)
    B, Hq, Hkv, Sq, Skv, D = _check_shapes(qa, ka, va)
    if da.shape != qa.shape:
        raise ValueError("dO must be shaped like Q")
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    dq = np.empty((B, Sq, Hq, D), dtype=np.float64)
    dk = np.empty((B, Skv, Hkv, D), dtype=np.float64)
    dv = np.empty((B, Skv, Hkv, D), dtype=np.float64)
    nt = lib.oracle_sdpa_bwd(qa.ctypes.data, ka.ctypes.data, va.ctypes.data, da.ctypes.data, DTYPES[dtype],
                             B, Hq, Hkv, Sq, Skv, D, float(scale), int(bool(causal)),
                             dq.ctypes.data, dk.ctypes.data, dv.ctypes.data, int(threads))
    if nt < 0:
        raise ValueError("oracle rejected the arguments")
    _last_threads = nt
    return dq, dk, dv


def last_threads() -> int:
    """Threads the most recent oracle call used."""
    return _last_threads


def max_threads() -> int:
    return load_library().oracle_max_threads()


def decode(codes, dtype: str, descale: float = 1.0) -> np.ndarray:
    """Decode raw element codes to float64 with the oracle's own decoders."""
    lib = load_library()
    a = _raw(codes, dtype).reshape(-1)
    code = DTYPES[dtype]
    return np.array([lib.oracle_decode(a.ctypes.data, i, code, float(descale)) for i in range(a.size)],
                    dtype=np.float64)


def row_index(b: int, i: int, hq: int, Sq: int, Hq: int) -> int:
    """Flat row index used by ``rows=``: (b*Sq + i)*Hq + hq."""
    return (b * Sq + i) * Hq + hq
