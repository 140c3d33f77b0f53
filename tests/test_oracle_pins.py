"""Pins for the fp64 attention oracle: each check comes from outside the oracle itself.

The oracle restates plain attention, which "Online Pseudo-average Shifting Attention (PASA)
for Robust Low-precision LLM Inference" (arXiv 2503.01873, Abstract) says PASA is
mathematically equivalent to. It is pinned here by a hand-worked example, by closed forms
(one key, two keys), by invariants (normalisation, constant values, shift invariance,
permutation equivariance, GQA = repeated-KV MHA) and by a library routine (PyTorch's fp64
scaled_dot_product_attention and logsumexp). A dropped max subtraction, a missing 1/l, a
wrong mask offset, a transposed operand or a wrong head mapping each fails at least one.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))


def f16(x):
    return np.asarray(x, dtype=np.float64).astype(np.float16)


def rand_inputs(rng, B, Hq, Hkv, Sq, Sk, D, scale=1.0):
    q = f16(rng.standard_normal((B, Hq, Sq, D)) * scale)
    k = f16(rng.standard_normal((B, Hkv, Sk, D)) * scale)
    v = f16(rng.standard_normal((B, Hkv, Sk, D)))
    return q, k, v


def torch_reference(q, k, v, causal, scale):
    """PyTorch fp64 SDPA with a bottom-right aligned causal mask (library routine)."""
    qt, kt, vt = (torch.from_numpy(x.astype(np.float64)) for x in (q, k, v))
    g = qt.shape[1] // kt.shape[1]
    kt = kt.repeat_interleave(g, dim=1)
    vt = vt.repeat_interleave(g, dim=1)
    Sq, Sk = qt.shape[2], kt.shape[2]
    mask = None
    if causal:
        mask = torch.ones(Sq, Sk, dtype=torch.bool).tril(diagonal=Sk - Sq)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    s = torch.matmul(qt, kt.transpose(-1, -2)) * scale
    if mask is not None:
        s = s.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    return o.numpy(), lse.numpy()


def test_half_decoder_matches_numpy(oracle_mod):
    # every finite binary16 pattern decodes to numpy's value; inf and NaN as such
    for bits in list(range(0, 65536, 97)) + [0x0001, 0x03FF, 0x0400, 0x7BFF, 0x7C00, 0xFC00, 0x8001]:
        ref = np.array([bits], np.uint16).view(np.float16).astype(np.float64)[0]
        got = oracle_mod.half_to_double(bits)
        if np.isnan(ref):
            assert np.isnan(got)
        else:
            assert got == ref, hex(bits)


@pytest.mark.parametrize("causal", [False, True])
def test_hand_worked_example(oracle_mod, causal):
    ex = json.load(open(os.path.join(HERE, "golden", "hand_example.json")))
    q, k, v = (f16(ex[n]) for n in ("q", "k", "v"))
    o, lse = oracle_mod.attention(q, k, v, causal=causal, scale=ex["scale"])
    ref = ex["causal" if causal else "noncausal"]
    np.testing.assert_allclose(o, np.array(ref["o"]), rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(lse, np.log(np.array(ref["lse_exp"], np.float64)), rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize(
    "B,Hq,Hkv,Sq,Sk,D,causal",
    [
        (1, 1, 1, 7, 7, 4, False),
        (1, 1, 1, 7, 7, 4, True),
        (2, 4, 2, 9, 13, 8, False),
        (2, 4, 2, 9, 13, 8, True),     # Sk > Sq: bottom-right aligned mask
        (1, 3, 1, 16, 5, 6, True),     # Sq > Sk: leading rows see no key
        (1, 6, 3, 33, 33, 16, True),
    ],
)
def test_matches_torch_sdpa_fp64(oracle_mod, B, Hq, Hkv, Sq, Sk, D, causal):
    rng = np.random.default_rng(B * 1000 + Sq * 10 + D)
    q, k, v = rand_inputs(rng, B, Hq, Hkv, Sq, Sk, D, scale=2.0)
    scale = 1.0 / math.sqrt(D)
    o, lse = oracle_mod.attention(q, k, v, causal=causal, scale=scale)
    o_ref, lse_ref = torch_reference(q, k, v, causal, scale)
    visible = np.isfinite(lse_ref)
    np.testing.assert_allclose(o[visible], o_ref[visible], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse[visible], lse_ref[visible], rtol=1e-12, atol=1e-12)
    # rows with no visible key: O = 0, LSE = -inf
    assert np.all(o[~visible] == 0.0)
    assert np.all(np.isneginf(lse[~visible]))


def test_single_key_closed_form(oracle_mod):
    rng = np.random.default_rng(3)
    q, k, v = rand_inputs(rng, 1, 2, 1, 5, 1, 16)
    o, lse = oracle_mod.attention(q, k, v, causal=False, scale=0.25)
    for h in range(2):
        np.testing.assert_array_equal(o[0, h], np.broadcast_to(v[0, 0, 0].astype(np.float64), (5, 16)))
        dots = q[0, h].astype(np.float64) @ k[0, 0, 0].astype(np.float64)
        np.testing.assert_allclose(lse[0, h], 0.25 * dots, rtol=1e-14, atol=1e-14)


def test_two_keys_logistic(oracle_mod):
    # with two keys softmax is the logistic function of the score difference
    rng = np.random.default_rng(4)
    q, k, v = rand_inputs(rng, 1, 1, 1, 6, 2, 8, scale=3.0)
    sc = 0.3
    o, lse = oracle_mod.attention(q, k, v, causal=False, scale=sc)
    qq, kk, vv = (x[0, 0].astype(np.float64) for x in (q, k, v))
    s0, s1 = sc * qq @ kk[0], sc * qq @ kk[1]
    w0 = 1.0 / (1.0 + np.exp(s1 - s0))
    np.testing.assert_allclose(o[0, 0], w0[:, None] * vv[0] + (1 - w0)[:, None] * vv[1], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse[0, 0], np.maximum(s0, s1) + np.log1p(np.exp(-np.abs(s0 - s1))), rtol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_rows_of_p_sum_to_one_and_constant_v(oracle_mod, causal):
    rng = np.random.default_rng(5)
    q, k, _ = rand_inputs(rng, 1, 2, 2, 20, 20, 8, scale=4.0)
    ones = np.ones((1, 2, 20, 8), np.float16)
    o, _ = oracle_mod.attention(q, k, ones, causal=causal)
    np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-14)
    c = f16(np.broadcast_to(np.linspace(-3, 3, 8), (1, 2, 20, 8)))
    o, _ = oracle_mod.attention(q, k, c, causal=causal)
    np.testing.assert_allclose(o, np.broadcast_to(c.astype(np.float64), o.shape), rtol=1e-13, atol=1e-13)


def test_causal_first_row_is_first_value(oracle_mod):
    rng = np.random.default_rng(6)
    q, k, v = rand_inputs(rng, 2, 2, 1, 9, 9, 8)
    o, lse = oracle_mod.attention(q, k, v, causal=True)
    for b in range(2):
        for h in range(2):
            np.testing.assert_array_equal(o[b, h, 0], v[b, 0, 0].astype(np.float64))


def test_shift_invariance(oracle_mod):
    # softmax is invariant to adding q_i . b to every score of row i:
    # K + 1 b^T leaves O unchanged and moves LSE by scale * q_i . b
    rng = np.random.default_rng(7)
    q = f16(rng.integers(-4, 5, (1, 2, 12, 16)))
    k = f16(rng.integers(-8, 9, (1, 2, 12, 16)))
    v = f16(rng.standard_normal((1, 2, 12, 16)))
    b = rng.integers(-300, 300, 16).astype(np.float64)
    kb = f16(k.astype(np.float64) + b)        # exact: small integers
    assert np.all(kb.astype(np.float64) == k.astype(np.float64) + b)
    for causal in (False, True):
        o0, l0 = oracle_mod.attention(q, k, v, causal=causal, scale=0.125)
        o1, l1 = oracle_mod.attention(q, kb, v, causal=causal, scale=0.125)
        np.testing.assert_allclose(o1, o0, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(l1 - l0, 0.125 * (q.astype(np.float64) @ b), rtol=1e-12, atol=1e-9)


def test_key_permutation_equivariance(oracle_mod):
    rng = np.random.default_rng(8)
    q, k, v = rand_inputs(rng, 1, 2, 1, 10, 17, 8)
    perm = rng.permutation(17)
    o0, l0 = oracle_mod.attention(q, k, v, causal=False)
    o1, l1 = oracle_mod.attention(q, np.ascontiguousarray(k[:, :, perm]), np.ascontiguousarray(v[:, :, perm]), causal=False)
    np.testing.assert_allclose(o1, o0, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(l1, l0, rtol=1e-13)


def test_gqa_equals_repeated_kv_mha(oracle_mod):
    rng = np.random.default_rng(9)
    q, k, v = rand_inputs(rng, 2, 6, 2, 11, 11, 8)
    kr = np.ascontiguousarray(np.repeat(k, 3, axis=1))
    vr = np.ascontiguousarray(np.repeat(v, 3, axis=1))
    for causal in (False, True):
        o0, l0 = oracle_mod.attention(q, k, v, causal=causal)
        o1, l1 = oracle_mod.attention(q, kr, vr, causal=causal)
        np.testing.assert_array_equal(o0, o1)
        np.testing.assert_array_equal(l0, l1)


def test_row_subset_matches_full(oracle_mod):
    rng = np.random.default_rng(10)
    q, k, v = rand_inputs(rng, 2, 4, 2, 13, 13, 8)
    o, lse = oracle_mod.attention(q, k, v, causal=True)
    rows = np.array([0, 5, 12, 13, 40, 103], np.int64)
    os_, ls = oracle_mod.attention(q, k, v, causal=True, rows=rows)
    np.testing.assert_array_equal(os_, o.reshape(-1, 8)[rows])
    np.testing.assert_array_equal(ls, lse.reshape(-1)[rows])


def test_large_scores_stay_finite(oracle_mod):
    # scores far beyond the fp16 range (|q.k| ~ 1e6) are exact in fp64: O is a convex
    # combination of V rows and equals the shifted-by-constant problem
    q = f16(np.full((1, 1, 4, 8), 60.0))
    k = f16(np.concatenate([np.full((1, 1, 3, 8), 500.0), np.full((1, 1, 3, 8), 499.0)], axis=2))
    v = f16(np.arange(48, dtype=np.float64).reshape(1, 1, 6, 8))
    o, lse = oracle_mod.attention(q, k, v, causal=False, scale=1.0 / 480.0)
    # scores: 60*500*8/480 = 500 for keys 0-2 and 499 for keys 3-5
    w = np.array([1, 1, 1, math.exp(-1), math.exp(-1), math.exp(-1)])
    ref = (w / w.sum()) @ v[0, 0].astype(np.float64)
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(ref, (4, 8)), rtol=1e-13)
    np.testing.assert_allclose(lse[0, 0], 500.0 + math.log(w.sum()), rtol=1e-14)


def test_row_max_abs_score_brute_force(oracle_mod):
    rng = np.random.default_rng(11)
    q, k, _ = rand_inputs(rng, 1, 4, 2, 9, 9, 8, scale=30.0)
    for causal in (False, True):
        got = oracle_mod.row_max_abs_score(q, k, causal=causal)
        qt = np.repeat(k, 2, axis=1)
        s = np.abs(np.einsum("bhid,bhjd->bhij", q.astype(np.float64), qt.astype(np.float64)))
        if causal:
            s = np.where(np.tril(np.ones((9, 9), bool)), s, 0.0)
        np.testing.assert_allclose(got, s.max(-1), rtol=1e-15)


def test_block_max_abs_score_brute_force(oracle_mod):
    # per key block, max |q_i . k_j| over the (i, j) pairs the mask allows, by a dense numpy
    # product on a tiny causal GQA case with a ragged last block (Sk = 10, blocks of 4)
    rng = np.random.default_rng(41)
    q = rng.standard_normal((2, 4, 7, 8)).astype(np.float16)
    k = rng.standard_normal((2, 2, 10, 8)).astype(np.float16)
    for causal in (False, True):
        got = oracle_mod.block_max_abs_score(q, k, 4, causal)
        s = np.abs(q.astype(np.float64) @ np.repeat(k, 2, axis=1).astype(np.float64).transpose(0, 1, 3, 2))
        if causal:
            i = np.arange(7)[:, None]
            j = np.arange(10)[None, :]
            s = np.where(j <= i + 10 - 7, s, 0.0)
        want = np.stack([s[..., 0:4].max(axis=(2, 3)), s[..., 4:8].max(axis=(2, 3)), s[..., 8:10].max(axis=(2, 3))], -1)
        np.testing.assert_array_equal(got, want)
        # the largest block value of a head is the largest row value of the head
        np.testing.assert_array_equal(got.max(-1), oracle_mod.row_max_abs_score(q, k, causal).max(-1))


def test_block_max_abs_score_recovered_equals_raw_when_shift_is_exact(oracle_mod):
    from oracle import pseudo_average as pa

    rng = np.random.default_rng(42)
    q = rng.integers(-3, 4, (1, 2, 30, 16)).astype(np.float16)
    k = (rng.integers(-20, 21, (1, 1, 300, 16)) + rng.integers(-200, 200, (1, 1, 1, 16))).astype(np.float16)
    ks, means = pa.kshift(k, block_rows=128)
    raw = oracle_mod.block_max_abs_score(q, k, 128, False)
    np.testing.assert_array_equal(oracle_mod.block_max_abs_score(q, ks, 128, False, means=means), raw)
    assert (oracle_mod.block_max_abs_score(q, ks, 128, False) < 0.5 * raw).all()   # the bias is gone
