"""GPU parity of the strided entry points and the log-sum-exp output.

Layouts: contiguous BSHD, BHSD (the (B, N, T, H) layout section 4 of the
codelab "Attention on GPU (cuDNN and TransformerEngine)" transposes into) and
a padded BSHD buffer with spare heads, for Q, K, V and O independently.  The
LSE of row i is log(sum_j exp(s_ij)) over the keys the row sees, the log of
the softmax denominator of section 1; the oracle computes it in fp64.

LSE tolerances, from the arithmetic:
  * bf16 / fp16: the scores are fp32 sums of exact products, the row sum an
    fp32 sum of exp2 values with relative error about 2^-22 each (at most
    n 2^-24 for the summation, n <= 4096 here), so |LSE - ref| stays near
    3e-4 at worst; the test allows 1e-3.
  * E4M3: the row sum is taken over the E4M3-rounded weights (relative error
    <= 2^-4 for normal values; subnormal ones, < 2^-6, err by <= 2^-10 each
    against a sum of at least 56), so at S <= 1024 |LSE - ref| <=
    log(1 + 2^-4 + 1024 * 2^-10 / 56) < 8e-2.
"""
import numpy as np
import pytest
import torch

import oracle
from sdpa_inputs import make_qkv, sample_rows
from tests.parity import assert_close, to_np

pytestmark = pytest.mark.gpu

LSE_TOL = {"bf16": 1e-3, "fp16": 1e-3, "e4m3": 8e-2}


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


DEV = "cuda:0"


def place(t: torch.Tensor, layout: str, fill=0):
    """A [B, S, H, D] view of a device copy of t stored in `layout`."""
    B, S, H, D = t.shape
    if layout == "bshd":
        return t.to(DEV).contiguous()
    if layout == "bhsd":
        return t.permute(0, 2, 1, 3).contiguous().to(DEV).permute(0, 2, 1, 3)
    if layout == "padded":                       # two spare heads per row, 8 spare rows per batch
        buf = torch.full((B, S + 8, H + 2, D), fill, dtype=t.dtype, device=DEV) if t.dtype.is_floating_point \
            and t.element_size() > 1 else torch.zeros((B, S + 8, H + 2, D), dtype=t.dtype, device=DEV)
        buf[:, :S, :H] = t.to(DEV)
        return buf[:, :S, :H]
    raise ValueError(layout)


def empty_out(shape, dtype, layout):
    B, S, H, D = shape
    if layout == "bshd":
        return torch.empty(shape, dtype=dtype, device=DEV)
    if layout == "bhsd":
        return torch.empty((B, H, S, D), dtype=dtype, device=DEV).permute(0, 2, 1, 3)
    buf = torch.full((B, S + 8, H + 2, D), float("nan"), dtype=dtype, device=DEV)
    return buf[:, :S, :H]


def run_ex(x, causal, lay_in, lay_out, with_lse=True):
    from scaled_dot_product_05_gb300 import sdpa_fwd_ex, sdpa_fwd_fp8_ex
    q, k, v = (place(t, lay_in) for t in (x.q, x.k, x.v))
    B, Sq, Hq, D = x.q.shape
    out_dtype = torch.bfloat16 if x.dtype == "e4m3" else x.q.dtype
    o = empty_out(tuple(x.q.shape), out_dtype, lay_out)
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=DEV) if with_lse else None
    if x.dtype == "e4m3":
        dq, dk, dv = x.descales
        sdpa_fwd_fp8_ex(q, k, v, o, lse, descale_q=dq, descale_k=dk, descale_v=dv, causal=causal)
    else:
        sdpa_fwd_ex(q, k, v, o, lse, causal=causal)
    torch.cuda.synchronize()
    return o, lse


def check_lse(lse, ref_lse, dtype, what):
    got = lse.cpu().double().numpy()
    assert np.isfinite(got).all(), what
    err = float(np.abs(got - ref_lse).max())
    assert err <= LSE_TOL[dtype], f"{what}: LSE max_abs {err:.3e} > {LSE_TOL[dtype]}"


SHAPES = [(2, 4, 2, 300, 300, 128), (1, 4, 4, 200, 77, 64), (1, 8, 1, 129, 400, 128), (1, 4, 2, 260, 260, 32)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("lay_in", ["bshd", "bhsd", "padded"])
@pytest.mark.parametrize("lay_out", ["bshd", "bhsd", "padded"])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_layouts_and_lse_bf16(shape, lay_in, lay_out, causal):
    B, Hq, Hkv, Sq, Skv, D = shape
    x = make_qkv(300 + Sq + D, B, Hq, Hkv, Sq, Skv, D, "bf16")
    o, lse = run_ex(x, causal, lay_in, lay_out)
    ref, ref_lse = oracle.sdpa_reference(x.q, x.k, x.v, causal=causal, dtype="bf16", return_lse=True)
    assert_close(to_np(o), ref, "bf16", f"{shape} {lay_in}->{lay_out}")
    check_lse(lse, ref_lse, "bf16", f"{shape} {lay_in}->{lay_out}")


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_layouts_and_lse_fp16(causal):
    x = make_qkv(321, 2, 6, 3, 257, 390, 128, "fp16")
    o, lse = run_ex(x, causal, "bhsd", "padded")
    ref, ref_lse = oracle.sdpa_reference(x.q, x.k, x.v, causal=causal, dtype="fp16", return_lse=True)
    assert_close(to_np(o), ref, "fp16", "fp16 bhsd->padded")
    check_lse(lse, ref_lse, "fp16", "fp16 bhsd->padded")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_layouts_and_lse_fp8(D, causal):
    x = make_qkv(330 + D, 1, 4, 2, 300, 300, D, "e4m3")
    o, lse = run_ex(x, causal, "bhsd", "bhsd")
    ref, ref_lse = oracle.sdpa_reference(x.q, x.k, x.v, causal=causal, dtype="e4m3", descales=x.descales,
                                         return_lse=True)
    assert_close(to_np(o), ref, "e4m3", f"fp8 D={D}")
    check_lse(lse, ref_lse, "e4m3", f"fp8 D={D}")


def test_ex_matches_plain_entry_point_bitwise():
    # contiguous layouts and no LSE: the same kernel launch as sdpa_fwd
    from scaled_dot_product_05_gb300 import sdpa_fwd
    x = make_qkv(340, 2, 8, 2, 520, 520, 128, "bf16")
    o_ex, _ = run_ex(x, True, "bshd", "bshd", with_lse=False)
    o = sdpa_fwd(x.q.to(DEV), x.k.to(DEV), x.v.to(DEV), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o_ex, o)


def test_output_layout_changes_only_addresses():
    # O in BHSD or a padded buffer holds bit-identical values to BSHD, the LSE
    # is identical, and the padding of the padded buffer is left untouched
    x = make_qkv(341, 1, 8, 4, 384, 384, 64, "bf16")
    o1, l1 = run_ex(x, True, "bshd", "bshd")
    o2, l2 = run_ex(x, True, "bhsd", "bhsd")
    o3, l3 = run_ex(x, True, "padded", "padded")
    assert torch.equal(o1, o2.contiguous()) and torch.equal(o1, o3.contiguous())
    assert torch.equal(l1, l2) and torch.equal(l1, l3)
    base = o3.as_strided((1, 384 + 8, 8 + 2, 64), (o3.stride(0), o3.stride(1), o3.stride(2), 1))
    assert torch.isnan(base[:, :, 8:].float()).all() and torch.isnan(base[:, 384:].float()).all()


def test_lse_closed_form_zero_query():
    # Q = 0: every score is 0, so LSE = log(number of visible keys)
    x = make_qkv(342, 1, 2, 2, 300, 300, 128, "bf16")
    x.q.zero_()
    _, lse = run_ex(x, True, "bshd", "bshd")
    want = np.log(np.arange(300) + 1.0)
    got = lse.cpu().double().numpy()
    assert np.abs(got - want[None, None, :]).max() <= 1e-5


@pytest.mark.parametrize("D", [32, 64])
def test_two_tile_ctas_small_head_dim_bhsd_lse_sampled(D):
    # D <= 64 above the one-tile threshold (B=8, Hq=16, S=1000: 512 units of
    # two Q tiles), BHSD in and out, LSE; the small shapes above cover the
    # one-tile layout with every layout
    B, Hq, Hkv, S = 8, 16, 4, 1000
    x = make_qkv(350 + D, B, Hq, Hkv, S, S, D, "bf16")
    o, lse = run_ex(x, True, "bhsd", "bhsd")
    rows = sample_rows(3 + D, B, S, Hq, 600)
    ref, ref_lse = oracle.sdpa_reference(x.q, x.k, x.v, causal=True, dtype="bf16", rows=rows, return_lse=True)
    flat = to_np(o.contiguous()).reshape(-1, D)
    assert_close(flat[rows], ref, "bf16", f"two-tile d{D} bhsd")
    l = lse.cpu().double().numpy()
    got = np.array([l[r // (Hq * S), r % Hq, (r // Hq) % S] for r in rows])
    assert np.abs(got - ref_lse).max() <= LSE_TOL["bf16"]


def test_causal_gqa_4096_bhsd_lse_sampled():
    # the headline workload with BHSD layouts and the LSE, sampled rows
    B, Hq, Hkv, S, D = 2, 32, 8, 4096, 128
    x = make_qkv(2, B, Hq, Hkv, S, S, D, "bf16")
    o, lse = run_ex(x, True, "bhsd", "bhsd")
    rows = sample_rows(2, B, S, Hq, 400)
    ref, ref_lse = oracle.sdpa_reference(x.q, x.k, x.v, causal=True, dtype="bf16", rows=rows, return_lse=True)
    flat = to_np(o.contiguous()).reshape(-1, D)
    assert_close(flat[rows], ref, "bf16", "gqa 4096 bhsd")
    l = lse.cpu().double().numpy()
    got = np.array([l[r // (Hq * S), r % Hq, (r // Hq) % S] for r in rows])
    assert np.abs(got - ref_lse).max() <= LSE_TOL["bf16"]
