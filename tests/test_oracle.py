"""Pins for the fp64 oracle (CPU only).

Each pin checks the oracle against something other than itself: values worked
by hand from the codelab "Attention on GPU (cuDNN and TransformerEngine)"
(tests/golden/hand_cases.json), closed forms and invariants the definition in
its section 1 fixes, the causal asymmetry of section 7, the GQA/MQA
broadcasting of section 9, a library routine for the same definition
(torch's float64 CPU scaled_dot_product_attention), and the element formats'
own definitions.  ``test_mutants_are_caught`` plants plausible mistakes in a
copy of the oracle's C source and checks that some pin fails for each.
"""
import json
import math
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from sdpa_inputs import make_qkv

HERE = os.path.dirname(os.path.abspath(__file__))


def ref(lib, q, k, v, **kw):
    return oracle.sdpa_reference(q, k, v, lib=lib, **kw)


def rnd(seed, *shape):
    return np.random.default_rng(seed).standard_normal(shape)


# ---------------------------------------------------------------- pins ------

def pin_hand_cases(lib):
    with open(os.path.join(HERE, "golden", "hand_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        q = np.array(c["q"], dtype=np.float64)[None, :, None, :]
        k = np.array(c["k"], dtype=np.float64)[None, :, None, :]
        v = np.array(c["v"], dtype=np.float64)[None, :, None, :]
        o, lse = ref(lib, q, k, v, causal=c["causal"], scale=c["scale"], dtype="f64", return_lse=True)
        np.testing.assert_allclose(o[0, :, 0, :], np.array(c["o"]), rtol=0, atol=1e-12, err_msg=c["name"])
        np.testing.assert_allclose(lse[0, 0, :], np.array(c["lse"]), rtol=0, atol=1e-12, err_msg=c["name"])


def pin_lse_closed_forms(lib):
    # Q = 0: every visible score is 0, so log sum exp = log(number of visible keys)
    Sq, Skv = 9, 12
    q, k, v = np.zeros((1, Sq, 2, 8)), rnd(60, 1, Skv, 1, 8), rnd(61, 1, Skv, 1, 8)
    _, lse = ref(lib, q, k, v, causal=False, dtype="f64", return_lse=True)
    np.testing.assert_allclose(lse, np.full((1, 2, Sq), math.log(Skv)), rtol=0, atol=1e-14)
    _, lse = ref(lib, q, k, v, causal=True, dtype="f64", return_lse=True)
    want = np.log(np.minimum(np.arange(Sq) + 1, Skv))
    np.testing.assert_allclose(lse[0, 0], want, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[0, 1], want, rtol=0, atol=1e-14)
    # one key: the log sum exp is that key's score, scale * q . k
    q, k = rnd(62, 1, 3, 1, 4), rnd(63, 1, 1, 1, 4)
    _, lse = ref(lib, q, k, k, causal=False, scale=0.7, dtype="f64", return_lse=True)
    np.testing.assert_allclose(lse[0, 0], 0.7 * (q[0, :, 0, :] @ k[0, 0, 0, :]), rtol=0, atol=1e-14)
    # one key 80 above the rest: log sum exp = that score + log(1 + O(e^-80))
    q = np.zeros((1, 1, 1, 2)); q[0, 0, 0, 0] = 1.0
    k = np.zeros((1, 5, 1, 2)); k[0, 3, 0, 0] = 80.0
    _, lse = ref(lib, q, k, k, causal=False, scale=1.0, dtype="f64", return_lse=True)
    assert abs(lse[0, 0, 0] - 80.0) < 1e-30 + 5 * math.exp(-80)


def pin_lse_scipy_logsumexp(lib):
    # a library routine for the same quantity: scipy's logsumexp of the
    # masked score matrix (scores formed here with einsum)
    from scipy.special import logsumexp
    q, k, v = rnd(64, 2, 7, 4, 8), rnd(65, 2, 10, 2, 8), rnd(66, 2, 10, 2, 8)
    scale = 0.37
    for causal in (False, True):
        _, lse = ref(lib, q, k, v, causal=causal, scale=scale, dtype="f64", return_lse=True)
        kr = np.repeat(k, 2, axis=2)                       # query head h reads KV head h // 2
        s = np.einsum("bihd,bjhd->bhij", q, kr) * scale
        if causal:
            s = np.where(np.tril(np.ones((7, 10), dtype=bool))[None, None], s, -np.inf)
        np.testing.assert_allclose(lse, logsumexp(s, axis=-1), rtol=0, atol=1e-12)


def pin_single_key(lib):
    # one key: softmax of one score is 1, so O = V for every query row
    q, k, v = rnd(1, 2, 5, 4, 8), rnd(2, 2, 1, 2, 8), rnd(3, 2, 1, 2, 8)
    for causal in (False, True):
        o = ref(lib, q, k, v, causal=causal, dtype="f64")
        expect = np.repeat(np.repeat(v, 5, axis=1), 2, axis=2)
        np.testing.assert_allclose(o, expect, rtol=0, atol=1e-13)


def pin_constant_v(lib):
    q, k = rnd(4, 2, 33, 4, 16), rnd(5, 2, 40, 2, 16)
    v = np.full((2, 40, 2, 16), -1.75)
    for causal in (False, True):
        o = ref(lib, q, k, v, causal=causal, dtype="f64")
        np.testing.assert_allclose(o, -1.75, rtol=0, atol=1e-13)


def pin_zero_query_is_mean(lib):
    # Q = 0: all scores 0, weights uniform over the visible keys
    B, Sq, Skv, Hq, Hkv, D = 2, 19, 23, 4, 2, 8
    q = np.zeros((B, Sq, Hq, D))
    k, v = rnd(6, B, Skv, Hkv, D), rnd(7, B, Skv, Hkv, D)
    o = ref(lib, q, k, v, causal=False, dtype="f64")
    mean_all = v.mean(axis=1)                                     # [B, Hkv, D]
    for hq in range(Hq):
        np.testing.assert_allclose(o[:, :, hq, :], np.broadcast_to(mean_all[:, None, hq // 2, :], (B, Sq, D)),
                                   rtol=0, atol=1e-13)
    oc = ref(lib, q, k, v, causal=True, dtype="f64")
    csum = np.cumsum(v, axis=1)
    for i in range(Sq):
        n = min(i + 1, Skv)
        for hq in range(Hq):
            np.testing.assert_allclose(oc[:, i, hq, :], csum[:, n - 1, hq // 2, :] / n, rtol=0, atol=1e-13)


def pin_causal_first_and_last_rows(lib):
    # section 7: position 0 attends only to itself, the last to every position
    x = make_qkv(11, 2, 4, 4, 64, 64, 32, "bf16")
    oc = ref(lib, x.q, x.k, x.v, causal=True, dtype="bf16")
    on = ref(lib, x.q, x.k, x.v, causal=False, dtype="bf16")
    v0 = x.v[:, 0].double().numpy()
    np.testing.assert_array_equal(oc[:, 0], v0)
    np.testing.assert_allclose(oc[:, -1], on[:, -1], rtol=0, atol=1e-13)
    assert np.abs(oc[:, 0] - on[:, 0]).max() > 0.1


def pin_causal_rows_are_prefix_attention(lib):
    # causal row i (top-left lower triangle) equals unmasked attention over keys 0..i;
    # with Sq > Skv the rows past the last key see every key
    B, Sq, Skv, H, D = 1, 12, 9, 2, 4
    q, k, v = rnd(8, B, Sq, H, D), rnd(9, B, Skv, H, D), rnd(10, B, Skv, H, D)
    oc = ref(lib, q, k, v, causal=True, dtype="f64")
    for i in range(Sq):
        n = min(i + 1, Skv)
        o_pref = ref(lib, q[:, i:i + 1], k[:, :n], v[:, :n], causal=False, dtype="f64")
        np.testing.assert_allclose(oc[:, i], o_pref[:, 0], rtol=0, atol=1e-13)


def pin_gqa_equals_repeated_mha(lib):
    # section 9: KV heads broadcast to query-head groups; equal to MHA on KV
    # heads repeated in place (repeat_interleave)
    for Hkv in (1, 2, 4):
        x = make_qkv(20 + Hkv, 2, 8, Hkv, 48, 40, 16, "bf16")
        G = 8 // Hkv
        k_rep = x.k.repeat_interleave(G, dim=2)
        v_rep = x.v.repeat_interleave(G, dim=2)
        for causal in (False, True):
            og = ref(lib, x.q, x.k, x.v, causal=causal, dtype="bf16")
            om = ref(lib, x.q, k_rep, v_rep, causal=causal, dtype="bf16")
            np.testing.assert_array_equal(og, om)


def pin_key_permutation_invariance(lib):
    q, k, v = rnd(12, 1, 7, 2, 8), rnd(13, 1, 29, 2, 8), rnd(14, 1, 29, 2, 8)
    perm = np.random.default_rng(15).permutation(29)
    o1 = ref(lib, q, k, v, causal=False, dtype="f64")
    o2 = ref(lib, q, k[:, perm], v[:, perm], causal=False, dtype="f64")
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)


def pin_key_shift_invariance(lib):
    # adding one vector u to every key adds q.u to every score of a row: the
    # softmax is unchanged (also under the causal mask)
    q, k, v = rnd(16, 1, 10, 2, 8), rnd(17, 1, 10, 2, 8), rnd(18, 1, 10, 2, 8)
    u = rnd(19, 8) * 3.0
    for causal in (False, True):
        o1 = ref(lib, q, k, v, causal=causal, dtype="f64")
        o2 = ref(lib, q, k + u, v, causal=causal, dtype="f64")
        np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)


def pin_dominant_key_large_logits(lib):
    # one key's score beats every other by > 60 while all scores are ~1000:
    # weight of the rest < exp(-60); the max subtraction keeps it finite
    D, S = 4, 16
    k = rnd(21, 1, S, 1, D)
    k[0, 5, 0] = [10.0, 0.0, 0.0, 0.0]
    k[0, :, 0, 0] = np.clip(k[0, :, 0, 0], -1, 1)
    k[0, 5, 0, 0] = 10.0
    q = np.zeros((1, 1, 1, D))
    q[0, 0, 0, 0] = 110.0          # scores = 110*k[:,0]; key 5: 1100, others <= 110
    v = rnd(22, 1, S, 1, D)
    o = ref(lib, q, k, v, causal=False, scale=1.0, dtype="f64")
    np.testing.assert_allclose(o[0, 0, 0], v[0, 5, 0], rtol=0, atol=1e-20)


def pin_weights_rows_sum_to_one(lib):
    x = make_qkv(23, 2, 4, 2, 37, 53, 16, "bf16")
    rows = list(range(0, 2 * 37 * 4, 3))
    for causal in (False, True):
        _, w = ref(lib, x.q, x.k, x.v, causal=causal, dtype="bf16", rows=rows, return_weights=True)
        np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-14)
        assert (w >= 0).all()
        if causal:
            for r, row_w in zip(rows, w):
                i = (r // 4) % 37
                assert (row_w[i + 1:] == 0).all() and row_w[min(i, 52)] > 0


def pin_torch_sdpa_float64(lib):
    # independent library routine for the same definition
    for (B, Hq, Hkv, Sq, Skv, D, causal, seed) in [
            (2, 4, 4, 33, 33, 16, False, 30), (2, 4, 4, 33, 33, 16, True, 31),
            (1, 8, 2, 20, 45, 32, False, 32), (1, 8, 2, 45, 20, 32, True, 33),
            (2, 6, 1, 17, 17, 8, True, 34)]:
        x = make_qkv(seed, B, Hq, Hkv, Sq, Skv, D, "bf16")
        scale = 1.0 / math.sqrt(D) * 1.3
        o = ref(lib, x.q, x.k, x.v, causal=causal, scale=scale, dtype="bf16")
        G = Hq // Hkv
        qt = x.q.double().transpose(1, 2)
        kt = x.k.double().repeat_interleave(G, dim=2).transpose(1, 2)
        vt = x.v.double().repeat_interleave(G, dim=2).transpose(1, 2)
        if causal:
            mask = torch.ones(Sq, Skv, dtype=torch.bool).tril()
            t = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
        else:
            t = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
        np.testing.assert_allclose(o, t.transpose(1, 2).numpy(), rtol=0, atol=1e-12)


def pin_e4m3_descales(lib):
    # E4M3 inputs: the oracle decodes each code and multiplies by its tensor's
    # descale; equal to the f64 oracle on torch's own float8 -> float64 values
    x = make_qkv(40, 1, 4, 2, 24, 30, 16, "e4m3")
    dq, dk, dv = x.descales
    o8 = ref(lib, x.q, x.k, x.v, causal=True, dtype="e4m3", descales=x.descales)
    qf = x.q.to(torch.float64).numpy() * dq
    kf = x.k.to(torch.float64).numpy() * dk
    vf = x.v.to(torch.float64).numpy() * dv
    of = ref(lib, qf, kf, vf, causal=True, dtype="f64")
    np.testing.assert_allclose(o8, of, rtol=0, atol=1e-13)
    # V's descale is a pure output scale; Q's and K's only enter the scores
    o_v2 = ref(lib, x.q, x.k, x.v, causal=True, dtype="e4m3", descales=(dq, dk, 2 * dv))
    np.testing.assert_allclose(o_v2, 2 * o8, rtol=0, atol=1e-13)


def bwd(lib, q, k, v, do, **kw):
    return oracle.sdpa_backward_reference(q, k, v, do, lib=lib, **kw)


def pin_bwd_finite_differences(lib):
    # central differences of the forward oracle: d/dX sum(dO * O(Q, K, V)),
    # independent of every formula in the backward routine
    B, Hq, Hkv, S, D = 1, 2, 1, 5, 3
    q, k, v, do = rnd(80, B, S, Hq, D), rnd(81, B, S, Hkv, D), rnd(82, B, S, Hkv, D), rnd(83, B, S, Hq, D)
    for causal in (False, True):
        dq, dk, dv = bwd(lib, q, k, v, do, causal=causal, scale=0.9, dtype="f64")

        def loss(q_, k_, v_):
            return float((ref(lib, q_, k_, v_, causal=causal, scale=0.9, dtype="f64") * do).sum())

        h = 1e-6
        for x, g, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
            num = np.zeros_like(x)
            for idx in np.ndindex(*x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p, args_m = [q, k, v], [q, k, v]
                args_p[which], args_m[which] = xp, xm
                num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
            np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8)


def pin_bwd_torch_autograd(lib):
    # torch's float64 autograd of scaled_dot_product_attention, GQA by
    # repeating K and V (their gradients sum over each group)
    B, Hq, Hkv, Sq, Skv, D = 2, 4, 2, 9, 11, 8
    q, k, v, do = rnd(84, B, Sq, Hq, D), rnd(85, B, Skv, Hkv, D), rnd(86, B, Skv, Hkv, D), rnd(87, B, Sq, Hq, D)
    for causal in (False, True):
        dq, dk, dv = bwd(lib, q, k, v, do, causal=causal, scale=0.4, dtype="f64")
        qt = torch.tensor(q).transpose(1, 2).requires_grad_()
        kt = torch.tensor(k).transpose(1, 2).requires_grad_()
        vt = torch.tensor(v).transpose(1, 2).requires_grad_()
        kr, vr = kt.repeat_interleave(2, dim=1), vt.repeat_interleave(2, dim=1)
        mask = torch.ones(Sq, Skv, dtype=torch.bool).tril() if causal else None
        o = torch.nn.functional.scaled_dot_product_attention(qt, kr, vr, attn_mask=mask, scale=0.4)
        o.backward(torch.tensor(do).transpose(1, 2))
        np.testing.assert_allclose(dq, qt.grad.transpose(1, 2).numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dk, kt.grad.transpose(1, 2).numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dv, vt.grad.transpose(1, 2).numpy(), rtol=0, atol=1e-12)


def pin_bwd_closed_forms(lib):
    # constant V: O is constant in Q and K, so dQ = dK = 0 and dV_j = sum of
    # the weights times dO; one key: the softmax is 1, so dQ = dK = 0 and
    # dV = sum over rows (and grouped heads) of dO
    q, k, do = rnd(88, 1, 6, 2, 4), rnd(89, 1, 7, 1, 4), rnd(90, 1, 6, 2, 4)
    v = np.full((1, 7, 1, 4), 2.5)
    dq, dk, _ = bwd(lib, q, k, v, do, causal=True, dtype="f64")
    np.testing.assert_allclose(dq, 0, atol=1e-14)
    np.testing.assert_allclose(dk, 0, atol=1e-14)
    k1, v1 = rnd(91, 1, 1, 1, 4), rnd(92, 1, 1, 1, 4)
    dq, dk, dv = bwd(lib, q, k1, v1, do, causal=False, dtype="f64")
    np.testing.assert_allclose(dq, 0, atol=1e-14)
    np.testing.assert_allclose(dk, 0, atol=1e-14)
    np.testing.assert_allclose(dv[0, 0, 0], do.sum(axis=(0, 1, 2)), rtol=0, atol=1e-13)


PINS = [pin_hand_cases, pin_single_key, pin_constant_v, pin_zero_query_is_mean,
        pin_causal_first_and_last_rows, pin_causal_rows_are_prefix_attention,
        pin_gqa_equals_repeated_mha, pin_key_permutation_invariance, pin_key_shift_invariance,
        pin_dominant_key_large_logits, pin_weights_rows_sum_to_one, pin_torch_sdpa_float64,
        pin_e4m3_descales, pin_lse_closed_forms, pin_lse_scipy_logsumexp, pin_bwd_finite_differences,
        pin_bwd_torch_autograd, pin_bwd_closed_forms]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


# ------------------------------------------------------- element decoders ----

def test_decode_bf16_all_codes():
    codes = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16)
    got = oracle.decode(codes.view(torch.bfloat16), "bf16")
    want = codes.view(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    np.testing.assert_array_equal(got[ok], want[ok])


def test_decode_fp16_all_codes():
    codes = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16)
    got = oracle.decode(codes.view(torch.float16), "fp16")
    want = codes.view(torch.float16).double().numpy()
    np.testing.assert_array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    np.testing.assert_array_equal(got[ok], want[ok])


def test_decode_e4m3_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    got = oracle.decode(codes.view(torch.float8_e4m3fn), "e4m3")
    want = codes.view(torch.float8_e4m3fn).double().numpy()
    np.testing.assert_array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    np.testing.assert_array_equal(got[ok], want[ok])
    assert np.nanmax(got) == 448.0 and np.isnan(got).sum() == 2


def test_thread_count_does_not_change_result(oracle_lib):
    x = make_qkv(50, 2, 4, 2, 70, 70, 32, "bf16")
    o1 = ref(oracle_lib, x.q, x.k, x.v, causal=True, dtype="bf16", threads=1)
    o4 = ref(oracle_lib, x.q, x.k, x.v, causal=True, dtype="bf16", threads=4)
    np.testing.assert_array_equal(o1, o4)


def test_rows_match_full(oracle_lib):
    x = make_qkv(51, 2, 4, 1, 65, 65, 16, "fp16")
    full = ref(oracle_lib, x.q, x.k, x.v, causal=True, dtype="fp16")
    rows = [0, 5, 64, 100, 2 * 65 * 4 - 1]
    part = ref(oracle_lib, x.q, x.k, x.v, causal=True, dtype="fp16", rows=rows)
    flat = full.reshape(-1, 16)
    np.testing.assert_array_equal(part, flat[rows])


def test_lse_rows_match_full(oracle_lib):
    # the row mode's LSE is the whole pass's [B][Hq][Sq] entry of the same row
    x = make_qkv(52, 2, 4, 2, 33, 40, 16, "bf16")
    _, full = ref(oracle_lib, x.q, x.k, x.v, causal=True, dtype="bf16", return_lse=True)
    rows = [0, 7, 33 * 4 + 2, 2 * 33 * 4 - 1]
    _, part = ref(oracle_lib, x.q, x.k, x.v, causal=True, dtype="bf16", rows=rows, return_lse=True)
    for r, val in zip(rows, part):
        hq, i, b = r % 4, (r // 4) % 33, r // (4 * 33)
        assert val == full[b, hq, i]


def test_rejects_bad_arguments(oracle_lib):
    q = np.zeros((1, 4, 3, 8))
    k = np.zeros((1, 4, 2, 8))
    with pytest.raises(ValueError):
        ref(oracle_lib, q, k, k, causal=False, dtype="f64")


# ------------------------------------------------------------- mutants ------

MUTANTS = {
    "gqa_modulo_head": ("const long g = hq / G;", "const long g = hq % p->Hkv;"),
    "causal_sees_next_key": ("n_vis = i + 1;", "n_vis = i + 2;"),
    "scale_dropped": ("scores[j] = acc * p->scale;", "scores[j] = acc;"),
    "no_max_subtraction": ("scores[j] = exp(scores[j] - m);", "scores[j] = exp(scores[j]);"),
    "softmax_sign_flipped": ("scores[j] = exp(scores[j] - m);", "scores[j] = exp(m - scores[j]);"),
    "not_normalised": ("scores[j] /= denom;", "scores[j] /= (denom + 1.0);"),
    "v_read_at_query_row": ("acc += scores[j] * load_elem(p->V, bshd(b, j, g, d,",
                            "acc += scores[j] * load_elem(p->V, bshd(b, i % p->Skv, g, d,"),
    "q_k_transposed": ("double k = load_elem(p->K, bshd(b, j, g, d,",
                       "double k = load_elem(p->K, bshd(b, i % p->Skv, g, d,"),
    "e4m3_descale_ignored": ("return decode_e4m3(((const uint8_t *)base)[idx]) * descale;",
                             "return decode_e4m3(((const uint8_t *)base)[idx]);"),
    "e4m3_bias_off_by_one": ("v = ldexp((double)(8 + f), e - 10);", "v = ldexp((double)(8 + f), e - 9);"),
    "fp16_subnormal_scale": ("v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    "lse_without_max": ("*lse_out = m + log(denom);", "*lse_out = log(denom);"),
    "lse_in_log2": ("*lse_out = m + log(denom);", "*lse_out = m + log2(denom);"),
    "bwd_causal_sees_next_key": ("? i + 1 : Skv;", "? i + 2 : Skv;"),
    "bwd_no_delta": ("const double dS = P[j] * (dP[j] - mean);", "const double dS = P[j] * dP[j];"),
    "bwd_dk_unscaled": ("dk[d] += scale * dS *", "dk[d] += dS *"),
    "bwd_dv_uses_ds": ("dv[d] += P[j] * load_elem(dO,", "dv[d] += dS * load_elem(dO,"),
    "bwd_dq_reads_v": ("dq[d] += scale * dS * load_elem(K, bshd(b, j, g, d,",
                       "dq[d] += scale * dS * load_elem(V, bshd(b, j, g, d,"),
}


def _build_mutant(tmp_path, name, old, new):
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, f"mutant {name}: pattern not unique"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    out = tmp_path / f"lib{name}.so"
    oracle.build(force=True, src=str(path), out=str(out))
    return oracle.load_library(str(out))


def _decoder_pins(lib):
    for dtype, codes in (("fp16", torch.arange(0, 1024, dtype=torch.int32).to(torch.int16).view(torch.float16)),
                         ("e4m3", torch.arange(0, 127, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn))):
        a = oracle._raw(codes, dtype)
        got = np.array([lib.oracle_decode(a.ctypes.data, i, oracle.DTYPES[dtype], 1.0) for i in range(a.size)])
        np.testing.assert_array_equal(got, codes.double().numpy())


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc needed to build mutants")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutants_are_caught(name, tmp_path):
    old, new = MUTANTS[name]
    lib = _build_mutant(tmp_path, name, old, new)
    caught = []
    for pin in PINS + [_decoder_pins]:
        try:
            with np.errstate(all="ignore"):
                pin(lib)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches mutant {name}"
