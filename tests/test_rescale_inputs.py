"""CPU check of the inputs of the GPU rescale test (tests/test_parity.py,
test_growing_max_rescales_every_tile): on them every row's running max
crosses the kernel's lazy-rescale threshold on every key tile, so that test
runs the rescale path (O and l times 2^(m_old - m_new) in TMEM) on every tile
after the first."""
import math

import pytest
import torch

from tests.parity import GROWING, growing_inputs


@pytest.mark.parametrize("shape,dtype", GROWING, ids=lambda v: "x".join(map(str, v)) if isinstance(v, tuple) else v)
def test_growing_max_inputs_cross_the_rescale_threshold(shape, dtype):
    # CPU: on these inputs every row's tile max (exp2 units, the kernel's
    # scale * log2 e) grows by more than the rescale threshold (8; 3 for
    # E4M3) from each full key tile to the next -- by more than 8 for all
    B, Hq, Hkv, Sq, Skv, D = shape
    x = growing_inputs(shape, dtype)
    dq, dk, _ = x.descales
    q = x.q.float().double() * dq          # E4M3 codes times their descale (1 for 16-bit)
    k = (x.k.float().double() * dk).repeat_interleave(Hq // Hkv, dim=2)
    s = torch.einsum("bihd,bjhd->bhij", q, k) / math.sqrt(D) / math.log(2.0)
    nt = Skv // 128
    tile_max = s[..., :nt * 128].reshape(B, Hq, Sq, nt, 128).amax(-1)
    assert (tile_max[..., 1:] - tile_max[..., :-1]).min().item() > 8.0
