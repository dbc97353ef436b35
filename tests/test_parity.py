"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs, element by element at sizes the oracle finishes in
seconds, and on sampled rows at the full benchmark sizes."""
import zlib

import numpy as np
import pytest
import torch

import oracle
from sdpa_inputs import make_qkv, sample_rows
from tests.parity import GROWING, assert_close, growing_inputs, to_np

pytestmark = pytest.mark.gpu


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


def run_gpu(x, causal, scale=None, stream=None):
    from scaled_dot_product_05_gb300 import sdpa_fwd
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in (x.q, x.k, x.v))
    o = sdpa_fwd(q, k, v, causal=causal, scale=scale, stream=stream)
    torch.cuda.synchronize()
    return o


# (B, Hq, Hkv, Sq, Skv, D): several tiles, ragged tails, Sq != Skv, tiny and
# degenerate shapes, MHA / GQA / MQA
SMALL = [
    (1, 2, 2, 128, 128, 64),
    (1, 2, 2, 128, 128, 128),
    (2, 4, 4, 384, 384, 64),
    (2, 4, 2, 256, 256, 128),
    (1, 8, 1, 300, 300, 128),
    (1, 4, 4, 200, 77, 64),
    (1, 4, 2, 77, 333, 128),
    (3, 1, 1, 129, 129, 64),
    (1, 1, 1, 1, 1, 128),
    (1, 2, 1, 1, 500, 64),
    (1, 2, 2, 500, 1, 128),
    (1, 6, 3, 640, 640, 128),
    (1, 6, 2, 300, 300, 128),      # 3 query heads per KV head: causal units of two tiles of one head
    (2, 8, 2, 1100, 1100, 128),    # causal, Sq > 1024: two tiles of one head even for an even group
    (2, 4, 2, 300, 300, 32),
    (1, 8, 8, 129, 520, 32),
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_small_full_compare(shape, causal, dtype):
    B, Hq, Hkv, Sq, Skv, D = shape
    x = make_qkv(zlib.crc32(repr((shape, causal, dtype)).encode()) % 100000, B, Hq, Hkv, Sq, Skv, D, dtype)
    o = run_gpu(x, causal)
    ref = oracle.sdpa_reference(x.q, x.k, x.v, causal=causal, dtype=dtype)
    assert_close(to_np(o), ref, dtype, f"{shape} causal={causal} {dtype}")


def test_explicit_scale_and_stream():
    x = make_qkv(77, 1, 4, 2, 256, 256, 128, "bf16")
    s = torch.cuda.Stream()
    o = run_gpu(x, True, scale=0.2, stream=s)
    ref = oracle.sdpa_reference(x.q, x.k, x.v, causal=True, scale=0.2, dtype="bf16")
    assert_close(to_np(o), ref, "bf16", "scale=0.2 side stream")


def test_causal_first_row_is_v0_and_last_row_matches_full():
    # section 7 of the codelab: position 0 sees only itself; the last sees all
    x = make_qkv(5, 2, 4, 4, 512, 512, 64, "bf16")
    oc, on = to_np(run_gpu(x, True)), to_np(run_gpu(x, False))
    np.testing.assert_array_equal(oc[:, 0], x.v[:, 0].double().numpy())
    assert np.abs(oc[:, -1] - on[:, -1]).max() <= 1e-2


def test_gqa_matches_repeated_kv_on_gpu():
    x = make_qkv(6, 1, 8, 2, 256, 256, 128, "bf16")
    o_g = run_gpu(x, True)
    x.k = x.k.repeat_interleave(4, dim=2).contiguous()
    x.v = x.v.repeat_interleave(4, dim=2).contiguous()
    o_m = run_gpu(x, True)
    assert torch.equal(o_g, o_m)


def test_deterministic():
    x = make_qkv(8, 2, 8, 2, 1024, 1024, 128, "bf16")
    a, b = run_gpu(x, True), run_gpu(x, True)
    assert torch.equal(a, b)


def test_tensor_map_cache_many_buffer_sets():
    # 1100 sets of Q, K, V, O buffers (4400 tensor maps, more than the
    # library's per-thread cache holds), cycled twice: the second pass mixes
    # cache hits with evictions and re-encodes, and must reproduce the first
    # pass bit for bit; a few sets are also checked against the oracle
    from scaled_dot_product_05_gb300 import sdpa_fwd
    dev = torch.device("cuda:0")
    x = make_qkv(77, 1, 2, 1, 130, 130, 64, "bf16")
    base = [t.to(dev) for t in (x.q, x.k, x.v)]
    n = 1100
    # distinct buffers and outputs at the inputs' own scale: Q rolled along
    # the sequence, K and V copied
    sets = [(torch.roll(base[0], i % 130, dims=1), base[1].clone(), base[2].clone()) for i in range(n)]
    outs = [torch.empty_like(base[0]) for _ in range(n)]
    for i in range(n):
        sdpa_fwd(*sets[i], outs[i], causal=(i % 2 == 1))
    first = [o.clone() for o in outs]
    for i in range(n):
        outs[i].fill_(0)
        sdpa_fwd(*sets[i], outs[i], causal=(i % 2 == 1))
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(first, outs))
    for i in (0, 1, 777):
        q, k, v = (t.cpu() for t in sets[i])
        ref = oracle.sdpa_reference(q, k, v, causal=(i % 2 == 1), dtype="bf16")
        assert_close(to_np(outs[i]), ref, "bf16", f"set {i}")


def test_output_guard_bands_untouched():
    from scaled_dot_product_05_gb300 import sdpa_fwd
    x = make_qkv(9, 1, 2, 2, 200, 200, 128, "bf16")
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in (x.q, x.k, x.v))
    n = q.numel()
    buf = torch.full((n + 2 * 4096,), 12345.0, dtype=torch.bfloat16, device=dev)
    o = buf[4096:4096 + n].view(q.shape)
    sdpa_fwd(q, k, v, o, causal=True)
    torch.cuda.synchronize()
    assert (buf[:4096] == 12345.0).all() and (buf[4096 + n:] == 12345.0).all()
    ref = oracle.sdpa_reference(x.q, x.k, x.v, causal=True, dtype="bf16")
    assert_close(to_np(o), ref, "bf16", "guarded")


# ---- the workload shapes, full size ----------------------------------------

def sampled_check(x, causal, n_rows, seed, dtype="bf16"):
    B, Sq, Hq, D = x.q.shape
    o = to_np(run_gpu(x, causal)).reshape(-1, D)
    rows = sample_rows(seed, B, Sq, Hq, n_rows)
    ref = oracle.sdpa_reference(x.q, x.k, x.v, causal=causal, dtype=dtype, rows=rows)
    return assert_close(o[rows], ref, dtype, f"{tuple(x.q.shape)} causal={causal}")


def test_tiny_mha_noncausal_full():
    x = make_qkv(0, 1, 2, 2, 128, 128, 64, "bf16")
    o = run_gpu(x, False)
    ref = oracle.sdpa_reference(x.q, x.k, x.v, causal=False, dtype="bf16")
    assert_close(to_np(o), ref, "bf16", "tiny MHA")


def test_causal_mha_1024_full():
    x = make_qkv(1, 4, 16, 16, 1024, 1024, 64, "bf16")
    o = run_gpu(x, True)
    ref = oracle.sdpa_reference(x.q, x.k, x.v, causal=True, dtype="bf16")
    assert_close(to_np(o), ref, "bf16", "causal MHA S=1024")


@pytest.mark.parametrize("D", [32, 64, 128])
def test_latency_row_b4_t128_full(D):
    # the codelab's small timing problem (B=4, T=128, N=8 heads, section 8),
    # with the head sizes its "Next steps" suggest; non-causal
    x = make_qkv(7 + D, 4, 8, 8, 128, 128, D, "bf16")
    o = run_gpu(x, False)
    ref = oracle.sdpa_reference(x.q, x.k, x.v, causal=False, dtype="bf16")
    assert_close(to_np(o), ref, "bf16", f"b4 t128 d{D}")


@pytest.mark.parametrize("B", [1, 16])
def test_batch_sweep_t256_full(B):
    # the batch sweep at T=256 (section 8): smallest and largest batch
    x = make_qkv(100 + B, B, 8, 8, 256, 256, 64, "bf16")
    o = run_gpu(x, False)
    ref = oracle.sdpa_reference(x.q, x.k, x.v, causal=False, dtype="bf16")
    assert_close(to_np(o), ref, "bf16", f"batch {B}")


# At D <= 64 the 16-bit pass runs one Q tile per CTA (two CTAs per SM) when
# units of two Q tiles would fill at most two rounds of the SMs (304 units on
# 152 SMs), else two Q tiles per CTA.  The shapes above are all below that
# line; these (B=8, Hq=16, S=1000: 512 two-tile units, ragged last tile, GQA
# 4:1) are above it, so both layouts meet the oracle at D = 32 and 64 (the
# small shapes run both 16-bit kinds through the one-tile layout).
@pytest.mark.parametrize("D", [32, 64])
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
def test_two_tile_ctas_at_small_head_dims_sampled(D, causal):
    x = make_qkv(40 + D, 8, 16, 4, 1000, 1000, D, "bf16")
    sampled_check(x, causal, 1500, 50 + D)


# The running max grows by at least 11 (exp2 units; checked on these inputs)
# from each full key tile to the next, so every row takes the lazy rescale (O
# and l times 2^(m_old - m_new), taken when the max grows by more than 8) on
# every tile after its first: query component 0 is 4 and key j's component 0
# is 32 j / 128.  N(0,1) inputs seldom take that path.
@pytest.mark.parametrize("shape,dtype", GROWING, ids=lambda v: "x".join(map(str, v)) if isinstance(v, tuple) else v)
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_growing_max_rescales_every_tile(shape, dtype, causal):
    x = growing_inputs(shape, dtype)
    if dtype == "e4m3":
        o = run_gpu_fp8(x, causal)
        ref = oracle.sdpa_reference(x.q, x.k, x.v, causal=causal, dtype="e4m3", descales=x.descales)
    else:
        o = run_gpu(x, causal)
        ref = oracle.sdpa_reference(x.q, x.k, x.v, causal=causal, dtype=dtype)
    assert_close(to_np(o), ref, dtype, f"growing max {shape} causal={causal}")


def test_causal_gqa_4096_sampled():
    x = make_qkv(2, 2, 32, 8, 4096, 4096, 128, "bf16")
    sampled_check(x, True, 3000, 2)


@pytest.mark.parametrize("B,S", [(64, 512), (32, 1024), (16, 2048), (8, 4096), (4, 8192), (2, 16384)])
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
def test_mqa_sweep_sampled(B, S, causal):
    x = make_qkv(3 + S, B, 32, 1, S, S, 128, "bf16")
    sampled_check(x, causal, 600 if S >= 8192 else 1000, 3 + S)


# ---- FP8 E4M3 inputs, bf16 output -------------------------------------------

def run_gpu_fp8(x, causal, scale=None):
    from scaled_dot_product_05_gb300 import sdpa_fwd_fp8
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in (x.q, x.k, x.v))
    dq, dk, dv = x.descales
    o = sdpa_fwd_fp8(q, k, v, descale_q=dq, descale_k=dk, descale_v=dv, causal=causal, scale=scale)
    torch.cuda.synchronize()
    return o


FP8_SMALL = [
    (1, 2, 2, 128, 128, 128),
    (2, 4, 2, 384, 384, 128),
    (1, 8, 1, 300, 300, 128),
    (1, 4, 4, 200, 77, 128),
    (1, 2, 2, 128, 128, 64),
    (2, 4, 2, 333, 333, 64),
]


@pytest.mark.parametrize("shape", FP8_SMALL, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_fp8_small_full_compare(shape, causal):
    B, Hq, Hkv, Sq, Skv, D = shape
    x = make_qkv(zlib.crc32(repr((shape, causal, "e4m3")).encode()) % 100000, B, Hq, Hkv, Sq, Skv, D, "e4m3")
    o = run_gpu_fp8(x, causal)
    assert o.dtype == torch.bfloat16
    ref = oracle.sdpa_reference(x.q, x.k, x.v, causal=causal, dtype="e4m3", descales=x.descales)
    assert_close(to_np(o), ref, "e4m3", f"fp8 {shape} causal={causal}")


def test_fp8_constant_v_is_returned():
    # the E4M3 weights are normalised by their own sum: constant V comes back
    # (up to the f16 partial sums and the bf16 output rounding)
    x = make_qkv(91, 1, 4, 2, 256, 256, 128, "e4m3")
    x.v = torch.full_like(x.v.view(torch.uint8), 0x3c).view(torch.float8_e4m3fn)   # 1.5
    o = to_np(run_gpu_fp8(x, True))
    assert np.abs(o - 1.5 * x.descales[2]).max() <= 4e-3 * 1.5 * x.descales[2] + 1e-6


def test_fp8_causal_8192_sampled():
    x = make_qkv(4, 2, 16, 16, 8192, 8192, 128, "e4m3")
    B, Sq, Hq, D = x.q.shape
    o = to_np(run_gpu_fp8(x, True)).reshape(-1, D)
    rows = sample_rows(4, B, Sq, Hq, 2000)
    ref = oracle.sdpa_reference(x.q, x.k, x.v, causal=True, dtype="e4m3", descales=x.descales, rows=rows)
    assert_close(o[rows], ref, "e4m3", "fp8 causal S=8192")
