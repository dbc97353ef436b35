"""ctypes view of the C ABI in include/sdpa.h (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB_PATH

SDPA_DTYPE_BF16, SDPA_DTYPE_FP16, SDPA_DTYPE_E4M3 = 0, 1, 2
STATUS = {0: "SDPA_OK", 1: "SDPA_ERR_NULL_PTR", 2: "SDPA_ERR_MISALIGNED", 3: "SDPA_ERR_BAD_SHAPE",
          4: "SDPA_ERR_HEADS", 5: "SDPA_ERR_HEAD_DIM", 6: "SDPA_ERR_DTYPE", 7: "SDPA_ERR_SCALE",
          8: "SDPA_ERR_ARCH", 9: "SDPA_ERR_ALIAS", 10: "SDPA_ERR_CUDA", 11: "SDPA_ERR_LAYOUT",
          12: "SDPA_ERR_WORKSPACE"}
# every function include/sdpa.h declares
EXPORTS = ("sdpa_fwd", "sdpa_fwd_fp8", "sdpa_fwd_ex", "sdpa_fwd_fp8_ex", "sdpa_fwd_decode",
           "sdpa_fwd_decode_noalloc", "sdpa_decode_workspace_bytes", "sdpa_bwd", "sdpa_bwd_workspace_bytes", "sdpa_bwd_fp8", "sdpa_bwd_fp8_workspace_bytes", "sdpa_status_string", "sdpa_last_cuda_error", "sdpa_device_error",
           "sdpa_abi_version")


class Layout(ctypes.Structure):
    """sdpa_layout_t: element strides (batch, seq, head) of a [B][S][H][D]
    tensor whose last dimension is contiguous."""
    _fields_ = [("batch", ctypes.c_longlong), ("seq", ctypes.c_longlong), ("head", ctypes.c_longlong)]

_lock = threading.Lock()
_lib = None


class SdpaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


def _bind(lib):
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.sdpa_fwd.restype = i
    lib.sdpa_fwd.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp]
    lib.sdpa_fwd_fp8.restype = i
    lib.sdpa_fwd_fp8.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, f, f, f, f, i, vp]
    lp = ctypes.POINTER(Layout)
    lib.sdpa_fwd_ex.restype = i
    lib.sdpa_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, lp, lp, lp, lp, f, i, i, vp]
    lib.sdpa_fwd_fp8_ex.restype = i
    lib.sdpa_fwd_fp8_ex.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, lp, lp, lp, lp, f, f, f, f, i, vp]
    lib.sdpa_fwd_decode.restype = i
    lib.sdpa_fwd_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, lp, lp, lp, lp, f, i, vp, ctypes.c_size_t, vp]
    lib.sdpa_fwd_decode_noalloc.restype = i
    lib.sdpa_fwd_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, lp, lp, lp, lp, f, i, vp]
    lib.sdpa_bwd.restype = i
    lib.sdpa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp, ctypes.c_size_t, vp]
    lib.sdpa_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.sdpa_bwd_workspace_bytes.argtypes = [i, i, i, i]
    lib.sdpa_bwd_fp8.restype = i
    lib.sdpa_bwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, f, f, f, f, f, vp, vp,
                                 ctypes.c_size_t, vp]
    lib.sdpa_bwd_fp8_workspace_bytes.restype = ctypes.c_size_t
    lib.sdpa_bwd_fp8_workspace_bytes.argtypes = [i, i, i, i]
    lib.sdpa_decode_workspace_bytes.restype = ctypes.c_size_t
    lib.sdpa_decode_workspace_bytes.argtypes = [i, i, i, i, i, i]
    lib.sdpa_status_string.restype = ctypes.c_char_p
    lib.sdpa_status_string.argtypes = [i]
    lib.sdpa_last_cuda_error.restype = i
    lib.sdpa_last_cuda_error.argtypes = []
    lib.sdpa_device_error.restype = i
    lib.sdpa_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint)]
    lib.sdpa_abi_version.restype = i
    lib.sdpa_abi_version.argtypes = []
    return lib


def lib():
    """The loaded CUDA library.  Raises if it has not been built: there is no
    other implementation to fall back to."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"CUDA library not built ({LIB_PATH}); run "
                                  "`python -c 'import __graft_entry__ as g; g.build()'`")
            _lib = _bind(ctypes.CDLL(LIB_PATH))
        return _lib


def status_string(status: int) -> str:
    return lib().sdpa_status_string(int(status)).decode()


def check(status: int) -> None:
    if status != 0:
        msg = status_string(status)
        if status == 10:
            msg += f" (cudaError {lib().sdpa_last_cuda_error()})"
        raise SdpaError(status, msg)
