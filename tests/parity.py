"""Shared helpers for the GPU parity tests: error metrics and tolerances.

Tolerances (bf16 / fp16): max |O - R| <= 1e-2 and ||O - R||_2 / ||R||_2 <=
4e-3 against the fp64 oracle R on the same inputs; FP8: max |O - R| <= 6e-2.
The codelab "Attention on GPU (cuDNN and TransformerEngine)" compares its
fused bf16 backends with allclose(rtol=1e-2, atol=1e-2) (section 6, "Force
the cuDNN fused backend")."""
import numpy as np
import torch

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
