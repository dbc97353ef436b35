"""Shared helpers for the GPU parity tests: error metrics, tolerances, and
the inputs of the lazy-rescale test.

Tolerances (bf16 / fp16): max |O - R| <= 1e-2 and ||O - R||_2 / ||R||_2 <=
4e-3 against the fp64 oracle R on the same inputs; FP8: max |O - R| <= 6e-2.
The codelab "Attention on GPU (cuDNN and TransformerEngine)" compares its
fused bf16 backends with allclose(rtol=1e-2, atol=1e-2) (section 6, "Force
the cuDNN fused backend")."""
import numpy as np
import torch

from sdpa_inputs import QKV, make_qkv, quantise_e4m3

TOL = {"bf16": (1e-2, 4e-3), "fp16": (1e-2, 4e-3), "e4m3": (6e-2, None)}


def to_np(o: torch.Tensor) -> np.ndarray:
    return o.float().cpu().double().numpy()


def errors(got: np.ndarray, ref: np.ndarray):
    d = got - ref
    max_abs = float(np.abs(d).max()) if d.size else 0.0
    nr = float(np.linalg.norm(ref))
    rel_rms = float(np.linalg.norm(d) / nr) if nr > 0 else float(np.linalg.norm(d))
    return max_abs, rel_rms


def assert_close(got, ref, dtype, what=""):
    max_abs, rel_rms = errors(got, ref)
    tol_abs, tol_rms = TOL[dtype]
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    assert max_abs <= tol_abs, f"{what}: max_abs {max_abs:.3e} > {tol_abs}"
    if tol_rms is not None:
        assert rel_rms <= tol_rms, f"{what}: rel_rms {rel_rms:.3e} > {tol_rms}"
    return max_abs, rel_rms


# Inputs on which the online softmax's running max grows by more than the
# lazy-rescale threshold from every key tile to the next (see
# tests/test_rescale_inputs.py); query component 0 is 4, key j's component 0
# is 32 j / 128.
GROWING = [((1, 4, 2, 1024, 1024, 128), "bf16"), ((2, 4, 4, 700, 700, 64), "bf16"),
           ((1, 2, 1, 640, 900, 128), "fp16"), ((1, 8, 2, 300, 1000, 32), "bf16"),
           ((1, 4, 2, 768, 768, 128), "e4m3"), ((2, 4, 4, 500, 500, 64), "e4m3")]


def growing_inputs(shape, dtype):
    B, Hq, Hkv, Sq, Skv, D = shape
    x = make_qkv(900 + D + Sq, B, Hq, Hkv, Sq, Skv, D, "bf16" if dtype == "e4m3" else dtype)
    q, k = x.q.float(), x.k.float()
    q[..., 0] = 4.0
    k[..., 0] = (32.0 * torch.arange(Skv, dtype=torch.float32) / 128.0).view(1, Skv, 1)
    # V halved: with the weights on a few keys |O| approaches max |V| (~4.5),
    # where one 16-bit rounding unit of O is already near the absolute bound;
    # a rescale mistake would still err by the order of |O|
    v = x.v.float() * 0.5
    if dtype == "e4m3":
        (q8, dq), (k8, dk), (v8, dv) = quantise_e4m3(q), quantise_e4m3(k), quantise_e4m3(v)
        return QKV(q8, k8, v8, "e4m3", (dq, dk, dv))
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    x.q, x.k, x.v = q.to(tdt), k.to(tdt), v.to(tdt)
    return x
