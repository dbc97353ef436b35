"""The bounded device waits, made to run out on purpose (GPU).

A test-only build of the library (the same sources compiled with
SDPA_WAIT_TEST; not the product library) takes a device wait limit and a
K-ring position whose copy the forward producer leaves out.  With a copy left
out, the waits that depend on that key tile cannot complete: after the short
limit the kernel records the wait's code in the device error word, raises its
abort flag, drains what is in flight, frees TMEM and returns.  Nothing faults
or hangs.  The test checks the code, that the call ended long before the
product's 2 s limit would allow, and that the context stays usable: a normal
call right after it matches the oracle, in the test build and in the product
library.  (The codelab's convention, section 6 "Force the cuDNN fused
backend": a request that cannot be served is reported as an error, not
silently replaced.)"""
import ctypes
import math
import time

import numpy as np
import pytest
import torch

import oracle
from sdpa_inputs import make_qkv
from tests.parity import assert_close, to_np

pytestmark = pytest.mark.gpu

# codes of the waits that depend on the second key tile of a unit
S_ISSUER_K_FULL = 0x203                 # the S issuer waits for the K tile
SOFTMAX_S_FULL = {0x301, 0x302}         # a softmax warpgroup waits for its S
PV_P_FULL = {0x206, 0x207}              # a P V issuer waits for P
EXPECTED = {S_ISSUER_K_FULL} | SOFTMAX_S_FULL | PV_P_FULL


@pytest.fixture(scope="module")
def test_lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from scaled_dot_product_05_gb300 import _abi
    from scaled_dot_product_05_gb300 import build
    build.build()
    lib = _abi._bind(ctypes.CDLL(build.build_wait_test()))
    lib.sdpa_test_set_wait.restype = ctypes.c_int
    lib.sdpa_test_set_wait.argtypes = [ctypes.c_ulonglong, ctypes.c_int]
    torch.cuda.set_device(0)
    yield lib
    assert lib.sdpa_test_set_wait(2_000_000_000, -1) == 0


def _device_error(lib):
    code = ctypes.c_uint(0)
    assert lib.sdpa_device_error(ctypes.byref(code)) == 0
    return int(code.value)


def _fwd(lib, q, k, v, o, causal):
    B, Sq, Hq, D = q.shape
    _, Skv, Hkv, _ = k.shape
    return lib.sdpa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, Hq, Hkv, Sq, Skv, D,
                        ctypes.c_float(1 / math.sqrt(D)), int(causal), 0, None)


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_withheld_key_tile_times_out_with_its_code_and_the_next_call_is_correct(test_lib, causal):
    lib = test_lib
    # two units of 256 query rows, two key tiles each: every CTA withholds its
    # second K copy (ring position 1)
    x = make_qkv(4242, 1, 2, 2, 256, 256, 64, "bf16")
    q, k, v = (t.cuda() for t in (x.q, x.k, x.v))
    o = torch.zeros_like(q)
    assert _device_error(lib) == 0
    assert lib.sdpa_test_set_wait(10_000_000, 1) == 0            # 10 ms per wait
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    assert _fwd(lib, q, k, v, o, causal) == 0                    # the launch itself succeeds
    code = _device_error(lib)                                    # synchronises
    elapsed = time.perf_counter() - t0
    assert code in EXPECTED, f"device error word 0x{code:x}"
    assert elapsed < 1.0, f"the timed-out call took {elapsed:.3f} s"
    assert _device_error(lib) == 0                               # read and cleared
    # the context is usable: a normal call is oracle-correct (test build with
    # the product's limit and nothing withheld, then the product library)
    assert lib.sdpa_test_set_wait(2_000_000_000, -1) == 0
    ref = oracle.sdpa_reference(x.q, x.k, x.v, causal=causal, dtype="bf16")
    o2 = torch.empty_like(q)
    assert _fwd(lib, q, k, v, o2, causal) == 0
    assert _device_error(lib) == 0
    assert_close(to_np(o2), ref, "bf16")
    from scaled_dot_product_05_gb300 import sdpa_device_error, sdpa_fwd
    o3 = sdpa_fwd(q, k, v, causal=causal)
    torch.cuda.synchronize()
    assert sdpa_device_error() == 0
    assert torch.equal(o3, o2)
