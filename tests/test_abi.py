"""C ABI checks that need no GPU: the library builds and loads, exports every
function include/sdpa.h declares, and rejects bad arguments with the
documented status before any CUDA call.

The argument checks pass fake device addresses that nothing may dereference.
Where a CUDA device can be reached, a call whose arguments got past every
check (the contiguous-layout case below, or a check that regressed) would
launch a kernel on those addresses, so every such test skips there: they are
CPU-only by construction, not just by their marker."""
import ctypes
import math
import os
import re

import pytest
import torch

from scaled_dot_product_05_gb300 import _abi
from scaled_dot_product_05_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return _abi.lib()


@pytest.fixture
def fake(lib):
    """The library, for calls that pass fake device addresses: only where no
    GPU can be reached."""
    if torch.cuda.is_available():
        pytest.skip("fake device addresses are passed only where no GPU can be reached")
    return lib


def declared_functions():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names.update(re.findall(r"\b(sdpa_\w+)\s*\(", text))
    return sorted(names)


def test_exports_every_declared_function(lib):
    names = declared_functions()
    assert names, "no declarations found"
    for n in names:
        assert hasattr(lib, n), f"{n} declared but not exported"
    assert set(names) == set(_abi.EXPORTS)


def test_abi_version_and_strings(lib):
    assert lib.sdpa_abi_version() >= 1
    for code in range(13):
        s = lib.sdpa_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.sdpa_status_string(99).decode() == "unknown status"


# fake, never dereferenced, 16-byte aligned device addresses, far apart
QP, KP, VP, OP = 0x10000000, 0x20000000, 0x30000000, 0x40000000
GOOD = dict(B=2, Hq=8, Hkv=2, Sq=300, Skv=300, D=128, scale=1 / math.sqrt(128), causal=1, dtype=0)


def call(lib, q=QP, k=KP, v=VP, o=OP, **kw):
    a = dict(GOOD, **kw)
    return lib.sdpa_fwd(q, k, v, o, a["B"], a["Hq"], a["Hkv"], a["Sq"], a["Skv"], a["D"],
                        ctypes.c_float(a["scale"]), a["causal"], a["dtype"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), 1), (dict(k=None), 1), (dict(v=None), 1), (dict(o=None), 1),
    (dict(q=QP + 8), 2), (dict(o=OP + 2), 2),
    (dict(B=0), 3), (dict(Hq=0), 3), (dict(Hkv=0), 3), (dict(Sq=0), 3), (dict(Skv=0), 3), (dict(Sq=-5), 3),
    (dict(B=1 << 20, Hq=1 << 12), 3),
    (dict(Hq=6, Hkv=4), 4),
    (dict(D=16), 5), (dict(D=96), 5), (dict(D=256), 5), (dict(D=0), 5),
    (dict(dtype=2), 6), (dict(dtype=7), 6),
    (dict(scale=0.0), 7), (dict(scale=-1.0), 7), (dict(scale=float("inf")), 7), (dict(scale=float("nan")), 7),
    (dict(o=QP + 16), 9), (dict(o=VP - 64), 9),
])
def test_rejects_before_any_cuda_call(fake, kw, status):
    assert call(fake, **kw) == status


def test_fp8_entry_checks(fake):
    f = fake.sdpa_fwd_fp8
    s = ctypes.c_float
    assert f(QP, KP, VP, None, 1, 2, 2, 128, 128, 64, s(0.125), s(1), s(1), s(1), 0, None) == 1
    assert f(QP, KP, VP, OP, 1, 2, 2, 128, 128, 64, s(0.125), s(0.0), s(1), s(1), 0, None) == 7
    # E4M3 rows must hold at least 64 bytes: D = 32 is a 16-bit-only head size
    assert f(QP, KP, VP, OP, 1, 2, 2, 128, 128, 32, s(0.125), s(1), s(1), s(1), 0, None) == 5
    assert f(QP, KP, VP, OP, 1, 2, 2, 128, 128, 48, s(0.125), s(1), s(1), s(1), 0, None) == 5


def test_valid_call_without_gpu_reports_cuda_error(fake):
    st = call(fake)
    assert st == 10
    assert fake.sdpa_last_cuda_error() != 0


def test_binding_rejects_cpu_tensors():
    from scaled_dot_product_05_gb300 import sdpa_fwd
    q = torch.zeros(1, 128, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        sdpa_fwd(q, q, q)


# ------------------------------------------------------------- *_ex checks --

def call_ex(lib, q=QP, k=KP, v=VP, o=OP, lse=None, ql=None, kl=None, vl=None, ol=None, **kw):
    a = dict(GOOD, **kw)
    ref = lambda l: ctypes.byref(_abi.Layout(*l)) if l is not None else None
    return lib.sdpa_fwd_ex(q, k, v, o, lse, a["B"], a["Hq"], a["Hkv"], a["Sq"], a["Skv"], a["D"],
                           ref(ql), ref(kl), ref(vl), ref(ol), ctypes.c_float(a["scale"]), a["causal"],
                           a["dtype"], None)


D_, SQ, HQ, HKV = 128, 300, 8, 2
BSHD_Q = (SQ * HQ * D_, HQ * D_, D_)
BHSD_Q = (HQ * SQ * D_, D_, SQ * D_)


@pytest.mark.parametrize("kw,status", [
    (dict(ql=(BSHD_Q[0], BSHD_Q[1], 4)), 11),           # head stride of 8 bytes: not a multiple of 16
    (dict(kl=(0, HKV * D_, D_)), 11),                     # zero stride
    (dict(vl=(-1, HKV * D_, D_)), 11),                    # negative stride
    (dict(ql=(1 << 40, HQ * D_, D_)), 11),                # 2^41 bytes
    (dict(ol=(SQ * HQ * D_, D_, D_)), 11),                # O rows overlap: seq and head stride both D
    (dict(ol=(D_, HQ * D_, D_ * 2)), 11),                 # O batch entries overlap other rows
    (dict(lse=0x50000002), 2),                            # LSE not 4-byte aligned
    (dict(lse=OP + 4096), 9),                             # LSE inside O
    (dict(lse=QP), 9),                                    # LSE inside Q
    (dict(o=QP + 2 * (HQ * SQ * D_ * 2) - 64, ql=BHSD_Q), 9),   # O starts inside the BHSD span of Q
    (dict(dtype=2), 6),
    (dict(q=None), 1),
])
def test_ex_rejects_before_any_cuda_call(fake, kw, status):
    assert call_ex(fake, **kw) == status


def test_ex_contiguous_layout_is_the_default(fake):
    # explicit contiguous strides pass the same checks as NULL layouts: the
    # only failure left is the device (none here) or a CUDA error
    st_null = call_ex(fake)
    st_expl = call_ex(fake, ql=BSHD_Q, kl=(SQ * HKV * D_, HKV * D_, D_), vl=(SQ * HKV * D_, HKV * D_, D_),
                      ol=BSHD_Q)
    assert st_null == st_expl and st_null in (8, 10)


def test_fp8_ex_checks(fake):
    f = fake.sdpa_fwd_fp8_ex
    s = ctypes.c_float
    bad = ctypes.byref(_abi.Layout(128 * 2 * 64, 2 * 64, 8))    # 8-byte head stride
    assert f(QP, KP, VP, OP, None, 1, 2, 2, 128, 128, 64, bad, None, None, None,
             s(0.125), s(1), s(1), s(1), 0, None) == 11
    assert f(QP, KP, VP, OP, None, 1, 2, 2, 128, 128, 64, None, None, None, None,
             s(0.125), s(1), s(-1), s(1), 0, None) == 7


def call_decode(lib, ws=None, ws_bytes=0, **kw):
    a = dict(GOOD, **kw)
    return lib.sdpa_fwd_decode(QP, KP, VP, OP, None, a["B"], a["Hq"], a["Hkv"], 1, a["Skv"], a["D"],
                               None, None, None, None, ctypes.c_float(a["scale"]), a["dtype"], ws, ws_bytes, None)


@pytest.mark.parametrize("kw,status", [
    (dict(Hq=12, Hkv=4), 4),          # G = 3 does not divide the 128 rows of a tile
    (dict(Hq=8, Hkv=3), 4),           # not a multiple
    (dict(dtype=2), 6),               # E4M3 has no decode pass
    (dict(ws=0x50000008, ws_bytes=1 << 20), 12),   # workspace not 16-byte aligned
    (dict(D=48), 5),
])
def test_decode_rejects_before_any_cuda_call(fake, kw, status):
    assert call_decode(fake, **kw) == status


def test_decode_workspace_query_rejects_bad_sizes(lib):
    assert lib.sdpa_decode_workspace_bytes(0, 8, 2, 1, 1000, 128) == 0
    assert lib.sdpa_decode_workspace_bytes(1, 8, 3, 1, 1000, 128) == 0
    assert lib.sdpa_decode_workspace_bytes(1, 8, 2, 1, 1000, 96) == 0


def test_decode_noalloc_rejects_before_any_cuda_call(fake):
    s = ctypes.c_float
    f = fake.sdpa_fwd_decode_noalloc
    assert f(QP, KP, VP, OP, None, 1, 12, 4, 1, 1000, 128, None, None, None, None, s(0.1), 0, None) == 4
    assert f(None, KP, VP, OP, None, 1, 8, 2, 1, 1000, 128, None, None, None, None, s(0.1), 0, None) == 1
    assert f(QP, KP, VP, OP, None, 1, 8, 2, 1, 1000, 128, None, None, None, None, s(0.1), 2, None) == 6


# the backward entry points: fake, never dereferenced, device addresses far apart
BP = dict(q=0x10000000, k=0x20000000, v=0x30000000, o=0x40000000, do=0x50000000, lse=0x60000000,
          dq=0x70000000, dk=0x80000000, dv=0x90000000, ws=0xA0000000, amax=0xB0000000)
BGOOD = dict(B=2, Hq=8, Hkv=2, Sq=300, Skv=300, D=128, scale=1 / math.sqrt(128), causal=1)


def call_bwd(lib, ws_bytes=None, dtype=0, **kw):
    a = dict(BGOOD, **{k: v for k, v in kw.items() if k in BGOOD})
    ptr = dict(BP, **{k: v for k, v in kw.items() if k in BP})
    if ws_bytes is None:
        ws_bytes = lib.sdpa_bwd_workspace_bytes(a["B"], a["Hq"], a["Sq"], 128)
    return lib.sdpa_bwd(ptr["q"], ptr["k"], ptr["v"], ptr["o"], ptr["do"], ptr["lse"], ptr["dq"], ptr["dk"],
                        ptr["dv"], a["B"], a["Hq"], a["Hkv"], a["Sq"], a["Skv"], a["D"], ctypes.c_float(a["scale"]),
                        a["causal"], dtype, ptr["ws"], ws_bytes, None)


def call_bwd_fp8(lib, ws_bytes=None, descales=(0.01, 0.01, 0.01, 1e-3), scale_ds=1.0, **kw):
    a = dict(BGOOD, **{k: v for k, v in kw.items() if k in BGOOD})
    ptr = dict(BP, **{k: v for k, v in kw.items() if k in BP})
    if ws_bytes is None:
        ws_bytes = lib.sdpa_bwd_fp8_workspace_bytes(a["B"], a["Hq"], a["Sq"], 128)
    f = ctypes.c_float
    return lib.sdpa_bwd_fp8(ptr["q"], ptr["k"], ptr["v"], ptr["o"], ptr["do"], ptr["lse"], ptr["dq"], ptr["dk"],
                            ptr["dv"], a["B"], a["Hq"], a["Hkv"], a["Sq"], a["Skv"], a["D"], f(a["scale"]),
                            a["causal"], *(f(x) for x in descales), f(scale_ds), ptr["amax"], ptr["ws"], ws_bytes,
                            None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), 1), (dict(do=None), 1), (dict(lse=None), 1), (dict(dk=None), 1), (dict(ws=None), 1),
    (dict(do=BP["do"] + 8), 2), (dict(ws=BP["ws"] + 4), 2),
    (dict(Sq=0), 3), (dict(Hq=6, Hkv=4), 4), (dict(D=32), 5), (dict(D=96), 5), (dict(dtype=2), 6),
    (dict(scale=0.0), 7), (dict(ws_bytes=1024), 12),
    (dict(dq=BP["q"] + 16), 9), (dict(dk=BP["ws"] + 64), 9), (dict(dv=BP["dk"]), 9),
])
def test_bwd_rejects_before_any_cuda_call(fake, kw, status):
    assert call_bwd(fake, **kw) == status


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), 1), (dict(o=None), 1), (dict(do=None), 1), (dict(lse=None), 1), (dict(ws=None), 1),
    (dict(do=BP["do"] + 8), 2), (dict(amax=BP["amax"] + 2), 2), (dict(o=BP["o"] + 8), 2),
    (dict(Skv=0), 3), (dict(Hq=6, Hkv=4), 4), (dict(D=32), 5), (dict(D=256), 5),
    (dict(scale=float("nan")), 7), (dict(descales=(0.01, 0.0, 0.01, 1e-3)), 7),
    (dict(descales=(0.01, 0.01, 0.01, float("inf"))), 7), (dict(scale_ds=0.0), 7), (dict(scale_ds=-2.0), 7),
    (dict(ws_bytes=4096), 12),
    (dict(dq=BP["q"] + 16), 9), (dict(amax=BP["ws"] + 64), 9), (dict(dk=BP["dv"]), 9),
])
def test_bwd_fp8_rejects_before_any_cuda_call(fake, kw, status):
    assert call_bwd_fp8(fake, **kw) == status


def test_bwd_fp8_workspace_bytes():
    from scaled_dot_product_05_gb300 import bwd_fp8_workspace_bytes, bwd_workspace_bytes
    # the bf16 dQ accumulator, fp32 Delta per query row and head, one 16-byte amax word
    assert bwd_fp8_workspace_bytes(2, 32, 4096, 128) == 2 * 4096 * 32 * 128 * 2 + 2 * 32 * 4096 * 4 + 16
    assert bwd_fp8_workspace_bytes(2, 32, 4096, 128) < bwd_workspace_bytes(2, 32, 4096, 128)
    assert bwd_fp8_workspace_bytes(2, 32, 4096, 32) == 0
