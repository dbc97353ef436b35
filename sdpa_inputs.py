"""Seeded synthetic inputs for the attention forward pass.

Shared by the oracle-side and the CUDA-side callers (tests, smoke check and
benchmark); it holds none of the attention arithmetic.  The recipe follows the
codelab "Attention on GPU (cuDNN and TransformerEngine)": section 3 draws
Q, K and V i.i.d. from N(0, 1) in float32 in the (B, T, N, H) layout, section 6
casts them to bfloat16, and section 10 ("FP8") feeds the forward pass E4M3
values under a per-tensor scale taken from the absolute maximum (recipe margin
0, amax "max").

Generator: ``torch.Generator('cpu').manual_seed(seed)``, then ``randn`` float32
for Q, K, V in that order, then round-to-nearest-even to bf16 / fp16, or, for
E4M3, x * (448 / amax(|x|)) rounded to E4M3 with descale = amax / 448.
Upstream gradients dO for the backward pass: ``randn`` float32 from their own
seed, rounded to bf16 / fp16, or, in the recipe's gradient format E5M2,
x * (57344 / amax(|x|)) rounded to E5M2 with descale = amax / 57344.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

E4M3_MAX = 448.0
E5M2_MAX = 57344.0


@dataclass
class QKV:
    q: torch.Tensor          # [B, Sq, Hq, D] on the CPU
    k: torch.Tensor          # [B, Skv, Hkv, D]
    v: torch.Tensor          # [B, Skv, Hkv, D]
    dtype: str               # "bf16", "fp16" or "e4m3"
    descales: tuple          # per-tensor (q, k, v) descales; 1.0 unless e4m3

    @property
    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.q, self.k, self.v))


def quantise_e4m3(x: torch.Tensor):
    """x -> (E4M3 codes of x * 448 / amax|x|, descale amax / 448)."""
    amax = float(x.abs().max())
    s = torch.tensor(E4M3_MAX / amax, dtype=torch.float32)
    x8 = (x * s).to(torch.float8_e4m3fn)
    return x8, float(torch.tensor(amax / E4M3_MAX, dtype=torch.float32))


def make_qkv(seed: int, B: int, Hq: int, Hkv: int, Sq: int, Skv: int, D: int,
             dtype: str = "bf16") -> QKV:
    """Seeded N(0,1) Q, K, V in BSHD layout (CPU tensors)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    q = torch.randn((B, Sq, Hq, D), generator=g, dtype=torch.float32)
    k = torch.randn((B, Skv, Hkv, D), generator=g, dtype=torch.float32)
    v = torch.randn((B, Skv, Hkv, D), generator=g, dtype=torch.float32)
    if dtype == "bf16":
        return QKV(q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16), dtype, (1.0, 1.0, 1.0))
    if dtype == "fp16":
        return QKV(q.to(torch.float16), k.to(torch.float16), v.to(torch.float16), dtype, (1.0, 1.0, 1.0))
    if dtype == "e4m3":
        (q8, dq), (k8, dk), (v8, dv) = quantise_e4m3(q), quantise_e4m3(k), quantise_e4m3(v)
        return QKV(q8, k8, v8, dtype, (dq, dk, dv))
    raise ValueError(f"unknown dtype {dtype!r}")


def _quantise_e5m2(x: torch.Tensor):
    amax = float(x.abs().max())
    s = torch.tensor(E5M2_MAX / amax, dtype=torch.float32)
    x8 = (x * s).to(torch.float8_e5m2)
    return x8, float(torch.tensor(amax / E5M2_MAX, dtype=torch.float32))


def make_grad(seed: int, shape, dtype: str = "bf16"):
    """Seeded N(0,1) upstream gradient dO (CPU tensor) of ``shape``: a bf16 /
    fp16 tensor, or for "e5m2" the pair (E5M2 codes, descale)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    x = torch.randn(tuple(shape), generator=g, dtype=torch.float32)
    if dtype == "bf16":
        return x.to(torch.bfloat16)
    if dtype == "fp16":
        return x.to(torch.float16)
    if dtype == "e5m2":
        return _quantise_e5m2(x)
    raise ValueError(f"unknown dtype {dtype!r}")


def sample_rows(seed: int, B: int, Sq: int, Hq: int, n: int, tile: int = 128):
    """Seeded sample of flat output-row indices (b*Sq + i)*Hq + hq.

    Always includes, for a few (b, hq) pairs, the first row, the last row, the
    first and last row of the last query tile and rows on either side of every
    tile boundary in the first few tiles, then fills up to ``n`` with uniform
    random rows."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) + 7919)
    fixed = set()
    special_i = {0, 1, Sq - 1, max(0, Sq - 2), (Sq - 1) // tile * tile}
    for t in range(1, min(4, (Sq + tile - 1) // tile)):
        special_i.update({t * tile - 1, t * tile})
    pairs = {(0, 0), (B - 1, Hq - 1), (B // 2, Hq // 2)}
    for b, h in pairs:
        for i in special_i:
            if 0 <= i < Sq:
                fixed.add((b * Sq + i) * Hq + h)
    total = B * Sq * Hq
    rows = sorted(fixed)
    if n > len(rows):
        extra = torch.randint(0, total, (n - len(rows),), generator=g).tolist()
        rows = sorted(set(rows).union(extra))
    return rows
