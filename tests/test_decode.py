"""GPU parity of the decode-shaped pass (sdpa_fwd_decode): the query heads of
a KV head stacked into one tile, with and without the key range split across
units, against the fp64 oracle and its log-sum-exp.  The codelab "Attention
on GPU (cuDNN and TransformerEngine)" motivates GQA / MQA by the KV cache of
inference (section 9); the pass is the same attention as section 1's,
non-causal.  Tolerances as in tests/parity.py and tests/test_layout_lse.py."""
import numpy as np
import pytest
import torch

import oracle
from sdpa_inputs import make_qkv
from tests.parity import assert_close, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from scaled_dot_product_05_gb300 import build
    build.build()
    torch.cuda.set_device(0)
    yield
    from scaled_dot_product_05_gb300 import sdpa_device_error
    assert sdpa_device_error() == 0


def run_decode(x, split, lse=True, layout="bshd"):
    from scaled_dot_product_05_gb300 import decode_workspace_bytes, sdpa_fwd_decode
    B, Sq, Hq, D = x.q.shape
    _, Skv, Hkv, _ = x.k.shape
    if layout == "bhsd":
        q, k, v = (t.permute(0, 2, 1, 3).contiguous().to(DEV).permute(0, 2, 1, 3) for t in (x.q, x.k, x.v))
        o = torch.empty((B, Hq, Sq, D), dtype=x.q.dtype, device=DEV).permute(0, 2, 1, 3)
    else:
        q, k, v = (t.to(DEV) for t in (x.q, x.k, x.v))
        o = torch.empty_like(q)
    l = torch.empty((B, Hq, Sq), dtype=torch.float32, device=DEV) if lse else None
    ws = None
    if split:
        nb = decode_workspace_bytes(B, Hq, Hkv, Sq, Skv, D)
        ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=DEV)
    sdpa_fwd_decode(q, k, v, o, l, workspace=ws)
    torch.cuda.synchronize()
    return o, l


# (B, Hq, Hkv, Sq, Skv, D): G = 8 with one query row, G = 4 with 4 rows,
# 128 stacked rows exactly, MHA (G = 1), G = 64 with 320 rows (a second,
# half-used pair), D = 32, a key length that is not a multiple of 128
SHAPES = [
    (2, 8, 1, 1, 1000, 128),
    (3, 32, 8, 4, 3000, 128),
    (1, 16, 2, 16, 700, 64),
    (2, 8, 8, 3, 513, 128),
    (1, 64, 1, 5, 2100, 128),
    (1, 8, 2, 7, 1500, 32),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("split", [False, True], ids=["whole", "split"])
def test_decode_matches_oracle(shape, split):
    B, Hq, Hkv, Sq, Skv, D = shape
    x = make_qkv(500 + Sq + Skv, B, Hq, Hkv, Sq, Skv, D, "bf16")
    o, lse = run_decode(x, split)
    ref, ref_lse = oracle.sdpa_reference(x.q, x.k, x.v, causal=False, dtype="bf16", return_lse=True)
    assert_close(to_np(o), ref, "bf16", f"decode {shape} split={split}")
    err = float(np.abs(lse.cpu().double().numpy() - ref_lse).max())
    assert err <= 1e-3, f"LSE max_abs {err:.3e}"


def test_decode_fp16_bhsd():
    x = make_qkv(530, 2, 16, 4, 2, 2500, 128, "fp16")
    o, lse = run_decode(x, True, layout="bhsd")
    ref, ref_lse = oracle.sdpa_reference(x.q, x.k, x.v, causal=False, dtype="fp16", return_lse=True)
    assert_close(to_np(o), ref, "fp16", "decode fp16 bhsd")
    assert float(np.abs(lse.cpu().double().numpy() - ref_lse).max()) <= 1e-3


def test_decode_split_and_whole_agree_with_standard_path():
    # three ways to the same attention: the standard pass and the decode pass
    # whole and split agree within the bf16 tolerance of one another
    from scaled_dot_product_05_gb300 import sdpa_fwd
    x = make_qkv(531, 4, 32, 8, 1, 4000, 128, "bf16")
    o_std = sdpa_fwd(x.q.to(DEV), x.k.to(DEV), x.v.to(DEV), causal=False)
    o_whole, _ = run_decode(x, False, lse=False)
    o_split, _ = run_decode(x, True, lse=False)
    torch.cuda.synchronize()
    a, b, c = to_np(o_std), to_np(o_whole), to_np(o_split)
    assert np.abs(a - b).max() <= 1e-2 and np.abs(a - c).max() <= 1e-2


def test_decode_workspace_too_small_is_rejected():
    from scaled_dot_product_05_gb300 import SdpaError, decode_workspace_bytes, sdpa_fwd_decode
    x = make_qkv(532, 2, 16, 2, 1, 8192, 128, "bf16")
    need = decode_workspace_bytes(2, 16, 2, 1, 8192, 128)
    assert need > 0
    q, k, v = (t.to(DEV) for t in (x.q, x.k, x.v))
    o = torch.full_like(q, 7.0)
    ws = torch.empty(need - 16, dtype=torch.uint8, device=DEV)
    with pytest.raises(SdpaError) as e:
        sdpa_fwd_decode(q, k, v, o, workspace=ws)
    assert e.value.status == 12
    torch.cuda.synchronize()
    assert (o == 7.0).all()                      # nothing was launched


def test_decode_gqa_32k_full_size():
    # the decode benchmark workload: 8 sequences, 32 query / 8 KV heads, one
    # query row each, 32768 cached keys; every output row against the oracle
    x = make_qkv(533, 8, 32, 8, 1, 32768, 128, "bf16")
    o, lse = run_decode(x, True)
    ref, ref_lse = oracle.sdpa_reference(x.q, x.k, x.v, causal=False, dtype="bf16", return_lse=True)
    assert_close(to_np(o), ref, "bf16", "decode 32k")
    assert float(np.abs(lse.cpu().double().numpy() - ref_lse).max()) <= 1e-3
