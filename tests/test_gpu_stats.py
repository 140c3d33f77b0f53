"""GPU: the overflow diagnostic (pasa_attn_fwd_stats) against the fp64 oracle.

"Online Pseudo-average Shifting Attention (PASA) for Robust Low-precision LLM Inference"
(arXiv 2503.01873), Abstract: fp16 attention scores overflow (> 65504) under a large
sequence-dimension bias of K and under Q/K resonance; shifting each key block by its
pseudo-average keeps them in range. The diagnostic reports, per query row, the largest
|score| the score accumulator held and the largest recovered |S' + q.m|; the oracle gives
both in fp64 (row_max_abs_score on raw or shifted keys, row_max_abs_recovered).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_helpers import to_dev
from oracle import pseudo_average as pa

pytestmark = pytest.mark.gpu
FP16_MAX = 65504.0


def run_stats(q, k, v, causal, mode):
    import precision_flashattention_numerics_gb300 as pasa

    qt, kt, vt = to_dev(q, k, v)
    o, lse, stats = pasa.attn_fwd_stats(qt, kt, vt, causal=causal, mode=mode)
    pasa.check_device_error()
    return o, lse, stats.double().cpu().numpy()


def fp16_spacing(x):
    return 2.0 ** (np.floor(np.log2(np.maximum(x, 2.0 ** -14))) - 10)


def abs_dot_bound(q, k, causal):
    """max_j sum_d |q_id k_jd| over the visible keys of each row: a bound on every partial sum
    an fp16 score accumulator holds while it adds up q_i . k_j."""
    g = q.shape[1] // k.shape[1]
    qa = np.abs(q.astype(np.float64))
    ka = np.repeat(np.abs(k.astype(np.float64)), g, axis=1)
    a = qa @ ka.transpose(0, 1, 3, 2)
    if causal:
        Sq, Sk = q.shape[2], k.shape[2]
        mask = np.arange(Sk)[None, :] <= np.arange(Sq)[:, None] + (Sk - Sq)
        a = np.where(mask, a, 0.0)
    return a.max(axis=-1)


@pytest.mark.parametrize("mode", [0, 1, 2, 3])
def test_stats_small_ragged(mode):
    w = wl.Workload("st", 1, 4, 2, 333, 333, 128, True, "kbias", 321, (("bias_std", 20.0),))
    q, k, v = wl.make_inputs(w)
    o, lse, st = run_stats(q, k, v, True, mode)
    ks, means = pa.kshift_fast(k)
    raw = oracle.row_max_abs_score(q, k, True)
    shifted = oracle.row_max_abs_score(q, ks, True)
    recovered = oracle.row_max_abs_recovered(q, ks, means, pa.block_rows_for(128), True)
    acc_ref = shifted if mode in (0, 1) else raw
    rec_ref = recovered if mode in (0, 1) else raw
    if mode in (1, 3):  # fp32 accumulation of exact fp16 products
        np.testing.assert_allclose(st[..., 0], acc_ref, rtol=2e-6, atol=1e-3)
        np.testing.assert_allclose(st[..., 1], rec_ref, rtol=2e-6, atol=1e-3)
    else:
        # fp16 accumulator: the MMA rounds the running sum to fp16 once per 16-channel step
        # (D / 16 roundings), each at most half a spacing of a partial sum, and every partial
        # sum is bounded by sum_d |q_d k_d|
        kk = ks if mode == 0 else k
        tol = (q.shape[-1] // 16) * fp16_spacing(abs_dot_bound(q, kk, True))
        assert np.all(np.abs(st[..., 0] - acc_ref) <= tol)
        assert np.all(np.abs(st[..., 1] - rec_ref) <= tol + 4 * fp16_spacing(rec_ref))
    # the shift shrinks what the accumulator holds
    if mode in (0, 1):
        assert np.median(raw / np.maximum(st[..., 0], 1e-3)) > 3.0


def test_stats_show_the_overflow_and_its_absence():
    w = wl.WORKLOADS["resonance_hot_a48_b2h5_s9216_d64"]
    q, k, v = wl.make_inputs(w)
    rows = np.random.default_rng(0).integers(0, w.B * w.Hq * w.Sq, 64)
    raw = oracle.row_max_abs_score(q, k, w.causal, rows=rows)
    ks, _ = pa.kshift_fast(k)
    shifted = oracle.row_max_abs_score(q, ks, w.causal, rows=rows)
    # naive fp16 accumulation: the rows whose raw scores pass 65504 hold inf
    _, _, st2 = run_stats(q, k, v, w.causal, 2)
    got2 = st2.reshape(-1, 2)[rows, 0]
    assert np.all(np.isinf(got2[raw > 1.05 * FP16_MAX]))
    assert np.all(np.isfinite(got2[raw < 0.9 * FP16_MAX]))
    assert np.mean(raw > 1.05 * FP16_MAX) > 0.3
    # PASA fp16 accumulation: every row stays finite and below the limit, close to the oracle
    _, _, st0 = run_stats(q, k, v, w.causal, 0)
    assert np.all(np.isfinite(st0)) and st0[..., 0].max() < FP16_MAX
    got0 = st0.reshape(-1, 2)[rows]
    assert np.all(np.abs(got0[:, 0] - shifted) <= 4 * fp16_spacing(shifted))
    # and the recovered raw magnitude is the one the naive kernel could not hold
    assert np.all(np.abs(got0[:, 1] - raw) <= 1e-2 * raw + 64.0)


def block_abs_dot_bound(q, k, causal, bn=128):
    """Per key block, the max over visible (i, j) of sum_d |q_id k_jd| (bounds every partial
    sum an fp16 accumulator holds for that block): [B, Hq, ceil(Sk / bn)]."""
    g = q.shape[1] // k.shape[1]
    a = np.abs(q.astype(np.float64)) @ np.repeat(np.abs(k.astype(np.float64)), g, axis=1).transpose(0, 1, 3, 2)
    Sq, Sk = q.shape[2], k.shape[2]
    if causal:
        mask = np.arange(Sk)[None, :] <= np.arange(Sq)[:, None] + (Sk - Sq)
        a = np.where(mask, a, 0.0)
    nb = -(-Sk // bn)
    return np.stack([a[..., j * bn:(j + 1) * bn].max(axis=(2, 3)) for j in range(nb)], axis=-1)


@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4])
def test_block_stats_small_ragged(mode):
    import precision_flashattention_numerics_gb300 as pasa

    w = wl.Workload("bst", 1, 4, 2, 333, 333, 128, True, "kbias", 322, (("bias_std", 20.0),))
    q, k, v = wl.make_inputs(w)
    qt, kt, vt = to_dev(q, k, v)
    o, lse, st, bst = pasa.attn_fwd_stats(qt, kt, vt, causal=True, mode=mode, block_stats=True)
    pasa.check_device_error()
    bst = bst.double().cpu().numpy()
    st = st.double().cpu().numpy()
    ks, means = pa.kshift_fast(k)
    shifted = mode in (0, 1, 4)
    acc_ref = oracle.block_max_abs_score(q, ks if shifted else k, 128, True)
    rec_ref = oracle.block_max_abs_score(q, ks, 128, True, means=means) if shifted else acc_ref
    assert bst.shape == acc_ref.shape + (2,)
    # the per-block and per-row maxima are reductions of the same numbers
    np.testing.assert_array_equal(bst[..., 0].max(-1), st[..., 0].max(-1))
    np.testing.assert_array_equal(bst[..., 1].max(-1), st[..., 1].max(-1))
    if mode in (1, 3):
        np.testing.assert_allclose(bst[..., 0], acc_ref, rtol=2e-6, atol=1e-3)
        np.testing.assert_allclose(bst[..., 1], rec_ref, rtol=2e-6, atol=1e-3)
    else:
        tol = (q.shape[-1] // 16) * fp16_spacing(block_abs_dot_bound(q, ks if shifted else k, True))
        assert np.all(np.abs(bst[..., 0] - acc_ref) <= tol)
        assert np.all(np.abs(bst[..., 1] - rec_ref) <= tol + 4 * fp16_spacing(rec_ref))


def test_block_stats_tell_bias_from_resonance():
    # The two causes of fp16 overflow (Abstract): a sequence-dimension bias of K, which the
    # shift removes (shifted max << raw max per block), and Q/K resonance varying within a
    # block, which it does not (shifted max close to raw max).
    import precision_flashattention_numerics_gb300 as pasa

    cases = {
        "bias": wl.Workload("b", 1, 4, 2, 1024, 1024, 128, True, "kbias", 331, (("bias_std", 20.0),)),
        "resonance": wl.Workload("r", 1, 2, 2, 2048, 2048, 64, False, "resonance", 332,
                                 (("A", 30.0), ("freq", "uniform_pi"), ("noise_std", 0.5), ("phase_flip", True))),
    }
    ratio = {}
    for name, w in cases.items():
        q, k, v = wl.make_inputs(w)
        qt, kt, vt = to_dev(q, k, v)
        _, _, _, bst = pasa.attn_fwd_stats(qt, kt, vt, causal=w.causal, mode=1, block_stats=True)
        pasa.check_device_error()
        bst = bst.double().cpu().numpy()
        ratio[name] = np.median(bst[..., 0] / bst[..., 1])
    assert ratio["bias"] < 0.2, ratio
    assert ratio["resonance"] > 0.6, ratio
