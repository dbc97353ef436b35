"""GPU parity of the backward pass (sdpa_bwd) against the fp64 oracle's
gradients of sum(dO * O), on the same seeded bf16 / fp16 inputs.  The forward
pass that produces O and the LSE is the library's own (as in training).

Tolerance, from the arithmetic: the kernel rounds P to 16 bits before dV =
P^T dO and dS = P (dP - Delta) before dK and dQ (relative error <= 2^-9 for
bf16, 2^-11 for fp16, per term), takes Delta from the 16-bit O, and rounds the
outputs to 16 bits; these are independent per term, so each gradient's
relative RMS error over the tensor stays within a few rounding units u (u =
2^-9 bf16, 2^-11 fp16; measured: 1.2 u to 1.4 u).  The test allows a relative
RMS of 4 u and a max-abs error of 10 u (bf16) / 10 u (fp16) of the tensor's
largest magnitude."""
import numpy as np
import pytest
import torch

import oracle
from sdpa_inputs import make_qkv

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
TOL = {"bf16": (4 * 2.0 ** -9, 10 * 2.0 ** -9), "fp16": (4 * 2.0 ** -11, 10 * 2.0 ** -11)}


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


def run(shape, causal, dtype="bf16", seed=0):
    from scaled_dot_product_05_gb300 import sdpa_bwd, sdpa_fwd_ex
    B, Hq, Hkv, Sq, Skv, D = shape
    x = make_qkv(900 + seed, B, Hq, Hkv, Sq, Skv, D, dtype)
    do = make_qkv(950 + seed, B, Hq, Hkv, Sq, Skv, D, dtype).q
    q, k, v, g = (t.to(DEV) for t in (x.q, x.k, x.v, do))
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=DEV)
    sdpa_fwd_ex(q, k, v, o, lse, causal=causal)
    dq, dk, dv = sdpa_bwd(q, k, v, o, g, lse, causal=causal)
    torch.cuda.synchronize()
    ref = oracle.sdpa_backward_reference(x.q, x.k, x.v, do, causal=causal, dtype=dtype)
    return [t.float().cpu().double().numpy() for t in (dq, dk, dv)], ref


def check(got, ref, what, dtype="bf16"):
    rel_rms, max_frac = TOL[dtype]
    for name, a, r in zip(("dQ", "dK", "dV"), got, ref):
        assert np.isfinite(a).all(), f"{what} {name}: non-finite"
        rms = float(np.linalg.norm(a - r) / max(np.linalg.norm(r), 1e-30))
        mx = float(np.abs(a - r).max() / max(np.abs(r).max(), 1e-30))
        print(f"{what} {name}: rel_rms {rms:.2e} max/|ref|max {mx:.2e}")
        assert rms <= rel_rms, f"{what} {name}: rel_rms {rms:.3e}"
        assert mx <= max_frac, f"{what} {name}: max error {mx:.3e} of the largest magnitude"


# several key and query tiles, ragged tails, Sq != Skv (including key tiles no
# causal query reaches), MHA / GQA / MQA, D = 64 / 128
SHAPES = [
    (1, 2, 2, 128, 128, 64),
    (2, 4, 2, 300, 300, 128),
    (1, 8, 1, 200, 77, 64),
    (1, 4, 4, 77, 333, 128),
    (2, 2, 2, 513, 513, 128),
    (1, 16, 2, 384, 384, 128),     # 8 query heads per KV head: query tiles last-first, heads innermost
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_backward_matches_oracle(shape, causal):
    got, ref = run(shape, causal)
    check(got, ref, f"{shape} causal={causal}")


def test_backward_fp16():
    got, ref = run((2, 4, 2, 256, 256, 128), True, dtype="fp16", seed=3)
    check(got, ref, "fp16", "fp16")


def test_backward_gqa_4096_one_group():
    # the causal GQA S=4096 workload at full size; the oracle checks one KV
    # head's group (batch 1, query heads 8..11, KV head 2): the gradients of
    # a group depend only on its own heads
    from scaled_dot_product_05_gb300 import sdpa_bwd, sdpa_fwd_ex
    B, Hq, Hkv, S, D = 2, 32, 8, 4096, 128
    x = make_qkv(2, B, Hq, Hkv, S, S, D, "bf16")
    do = make_qkv(3, B, Hq, Hkv, S, S, D, "bf16").q
    q, k, v, g = (t.to(DEV) for t in (x.q, x.k, x.v, do))
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device=DEV)
    sdpa_fwd_ex(q, k, v, o, lse, causal=True)
    dq, dk, dv = sdpa_bwd(q, k, v, o, g, lse, causal=True)
    torch.cuda.synchronize()
    b, hk = 1, 2
    hs = slice(hk * 4, hk * 4 + 4)
    ref = oracle.sdpa_backward_reference(x.q[b:b + 1, :, hs].contiguous(), x.k[b:b + 1, :, hk:hk + 1].contiguous(),
                                         x.v[b:b + 1, :, hk:hk + 1].contiguous(), do[b:b + 1, :, hs].contiguous(),
                                         causal=True, dtype="bf16")
    got = [t.float().cpu().double().numpy() for t in (dq[b:b + 1, :, hs], dk[b:b + 1, :, hk:hk + 1],
                                                      dv[b:b + 1, :, hk:hk + 1])]
    check(got, ref, "gqa 4096 group")


def test_backward_deterministic_dk_dv():
    # dK and dV are reduced inside one CTA: bit-identical across runs
    from scaled_dot_product_05_gb300 import sdpa_bwd, sdpa_fwd_ex
    x = make_qkv(960, 1, 4, 2, 384, 384, 128, "bf16")
    q, k, v = (t.to(DEV) for t in (x.q, x.k, x.v))
    g = torch.randn(q.shape, device=DEV).to(q.dtype)
    o = torch.empty_like(q)
    lse = torch.empty((1, 4, 384), dtype=torch.float32, device=DEV)
    sdpa_fwd_ex(q, k, v, o, lse, causal=True)
    a = sdpa_bwd(q, k, v, o, g, lse, causal=True)
    b = sdpa_bwd(q, k, v, o, g, lse, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


# degenerate shapes: one query row, one key, exact tile multiples, B > 1 with
# one KV head.  Where every visible P is 1 (one key, or causal row 0) dS =
# dP - Delta = 0 and dQ, dK vanish up to rounding, so each error is taken
# relative to the largest gradient of the problem when its own is ~0.
EDGE = [(1, 2, 1, 1, 1, 64), (1, 2, 1, 1, 300, 128), (1, 2, 2, 300, 1, 64), (1, 4, 2, 256, 256, 128),
        (3, 2, 1, 129, 129, 64)]


def check_edge(got, ref, what, rel):
    scale = max(float(np.linalg.norm(r)) for r in ref)
    for name, a, r in zip(("dQ", "dK", "dV"), got, ref):
        assert np.isfinite(a).all(), f"{what} {name}: non-finite"
        err = float(np.linalg.norm(a - r)) / max(float(np.linalg.norm(r)), 1e-3 * scale)
        print(f"{what} {name}: rel {err:.3e}")
        assert err <= rel, f"{what} {name}: {err:.3e} > {rel}"


@pytest.mark.parametrize("shape", EDGE, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_backward_edge_shapes(shape, causal):
    got, ref = run(shape, causal, seed=7)
    check_edge(got, ref, f"{shape} causal={causal}", TOL["bf16"][0])
