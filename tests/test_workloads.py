"""Input generators, and the overflow facts the abstract states, checked with the oracle.

"Online Pseudo-average Shifting Attention (PASA) for Robust Low-precision LLM Inference"
(arXiv 2503.01873), Abstract: a large bias along the sequence dimension and Q/K resonance
(phase coincidence or a 180-degree phase shift) push attention scores past 65504, the
largest fp16 value; shifting each key block by its pseudo-average avoids the overflow.
"""
import numpy as np
import pytest

import workloads as wl
from oracle import pseudo_average as pa

FP16_MAX = 65504.0


def test_generators_are_deterministic_and_fp16():
    w = wl.WORKLOADS["iid_b1h1_s128_d64"]
    a = wl.make_inputs(w)
    b = wl.make_inputs(w)
    for x, y, shape in zip(a, b, [(1, 1, 128, 64)] * 3):
        assert x.dtype == np.float16 and x.shape == shape and x.flags.c_contiguous
        assert x.tobytes() == y.tobytes()
    c = wl.make_inputs(w, seed=5)
    assert c[0].tobytes() != a[0].tobytes()


def test_shapes_of_measured_workloads():
    shapes = {
        "iid_b1h1_s128_d64": (1, 1, 1, 128, 64, False),
        "kbias20_b1h28g4_s4096_d128_causal": (1, 28, 4, 4096, 128, True),
        "resonance_a30_b2h5_s9216_d64": (2, 5, 5, 9216, 64, False),
        "iid_b4h32g8_s8192_d128_causal": (4, 32, 8, 8192, 128, True),
        "kbias10_t3_b1h28g4_s32768_d128_causal": (1, 28, 4, 32768, 128, True),
    }
    assert list(shapes) == wl.MEASURED
    for name, (B, Hq, Hkv, S, D, causal) in shapes.items():
        w = wl.WORKLOADS[name]
        assert (w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, w.causal) == (B, Hq, Hkv, S, S, D, causal)
        assert w.scale == pytest.approx(D ** -0.5)


def test_flop_convention():
    w = wl.WORKLOADS["iid_b4h32g8_s8192_d128_causal"]
    S = 8192
    assert w.flops() == 4.0 * 4 * 32 * 128 * (S * (S + 1) // 2)
    w1 = wl.WORKLOADS["iid_b1h1_s128_d64"]
    assert w1.flops() == 4.0 * 128 * 128 * 64


def test_kbias_statistics():
    w = wl.WORKLOADS["kbias20_b1h28g4_s4096_d128_causal"]
    q, k, v = wl.make_inputs(w)
    kb = k.astype(np.float64)
    bias = kb.mean(axis=2)                       # per (b, kv-head, channel)
    assert 14 < bias.std() < 26                  # N(0, 20^2) bias
    assert abs((kb - bias[:, :, None, :]).std() - 1.0) < 0.02
    assert abs(q.astype(np.float64).std() - 1.0) < 0.01


def _sampled_max_scores(oracle_mod, w, n_rows=48):
    q, k, v = wl.make_inputs(w)
    rows = np.random.default_rng(0).integers(0, w.B * w.Hq * w.Sq, n_rows)
    raw = oracle_mod.row_max_abs_score(q, k, w.causal, rows=rows)
    ks, _ = pa.kshift_fast(k)
    shifted = oracle_mod.row_max_abs_score(q, ks, w.causal, rows=rows)
    return raw, shifted


def test_overflow_demo_raw_scores_overflow_shifted_do_not(oracle_mod):
    raw, shifted = _sampled_max_scores(oracle_mod, wl.WORKLOADS["resonance_hot_a48_b2h5_s9216_d64"])
    assert np.mean(raw > FP16_MAX) > 0.5     # most rows hold a score beyond the fp16 range
    assert shifted.max() < FP16_MAX / 2      # after the shift none comes close


def test_kbias_shift_shrinks_scores(oracle_mod):
    raw, shifted = _sampled_max_scores(oracle_mod, wl.WORKLOADS["kbias20_b1h28g4_s4096_d128_causal"])
    assert np.median(raw / shifted) > 3.0
    assert raw.max() / shifted.max() > 5.0


def test_literal_resonance_stays_below_fp16_max(oracle_mod):
    # with A = 30, D = 64: |q.k| <= A^2 D + noise = 57600 + O(100) < 65504; the shift cannot
    # shrink resonance that varies within one key block (mean ~ 0)
    raw, shifted = _sampled_max_scores(oracle_mod, wl.WORKLOADS["resonance_a30_b2h5_s9216_d64"])
    assert raw.max() < FP16_MAX
    assert raw.max() > 5000.0
