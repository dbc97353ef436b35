"""The benchmark's FLOP and algorithmic-byte counts, which every roofline
fraction divides by, checked against counts made by hand for each kind of
workload (CPU only)."""
import pytest

import bench


def test_headline_forward_counts():
    # causal GQA B=2 Hq=32 Hkv=8 S=4096 D=128 bf16: 4 D FLOPs per visible
    # score, half the S x S scores; Q and O are 2 x 4096 x 32 x 128 x 2 bytes,
    # K and V 2 x 4096 x 8 x 128 x 2 bytes
    assert bench.step_flops("gqa-causal-4096") == 4 * 2 * 32 * 4096 * 4096 * 128 / 2
    q = 2 * 4096 * 32 * 128 * 2
    kv = 2 * 4096 * 8 * 128 * 2
    assert bench.step_bytes("gqa-causal-4096") == 2 * q + 2 * kv == 167772160


def test_fp8_forward_counts():
    # E4M3 Q, K, V (one byte), bf16 O; MHA B=2 H=16 S=8192 D=128
    n = 2 * 8192 * 16 * 128
    assert bench.step_bytes("fp8-causal-8192") == n * (1 + 1 + 1 + 2)
    assert bench.step_flops("fp8-causal-8192") == 4 * 2 * 16 * 8192 * 8192 * 128 / 2


def test_decode_counts():
    # decode pass, non-causal, B=8 Hq=32 Hkv=8 Sq=1 Skv=32768 D=128: K and V
    # dominate (1.07 GB), every score visible
    q = 8 * 1 * 32 * 128 * 2
    kv = 8 * 32768 * 8 * 128 * 2
    assert bench.step_bytes("decode-gqa-b8-32k") == 2 * q + 2 * kv
    assert bench.step_flops("decode-gqa-b8-32k") == 4 * 8 * 32 * 1 * 32768 * 128


@pytest.mark.parametrize("name,e", [("bwd-gqa-causal-4096", 2), ("bwd-fp8-causal-8192", 1)])
def test_backward_counts(name, e):
    # five products of 2 D FLOPs per visible score; Q, dO (e bytes), O, dQ
    # (2 bytes) per query row and head, K, V (e bytes), dK, dV (2 bytes) per
    # key row and KV head, the fp32 LSE per query row and head
    w = bench.spec(name)
    visible = w.B * w.Hq * w.Sq * w.Skv / (2 if w.causal else 1)
    assert bench.step_flops(name) == 10 * w.D * visible
    rows_q = w.B * w.Sq * w.Hq
    rows_k = w.B * w.Skv * w.Hkv
    want = rows_q * w.D * (e + e + 2 + 2) + rows_k * w.D * (e + e + 2 + 2) + 4 * rows_q
    assert bench.step_bytes(name) == want
