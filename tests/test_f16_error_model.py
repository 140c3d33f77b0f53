"""CPU check of the error model behind the fp16-score gates of the GPU tests.

The GPU tests gate the fp16-accumulated score modes (0, 2, 4) on the resonance and biased
workloads with f16_score_rmse_model (tests/gpu_helpers.py): a first-order propagation of
round-to-nearest errors of an fp16 accumulator, one rounding per 16-channel MMA step. Here
that prediction is compared with a direct emulation of such an accumulator in numpy: the
exact 16-channel partial dot products of the fp16 inputs are added to an fp16 accumulator
with one round-to-nearest-even each, the recovered scores are formed in fp64 and the
softmax is taken in fp64. The gate built on the model (F16_MODEL_FACTOR x the prediction)
must pass such an accumulator, and the prediction must not be vacuous, on the input families of the measured workloads ("Online Pseudo-average
Shifting Attention (PASA) for Robust Low-precision LLM Inference", Abstract: the two
overflow causes, sequence-dimension bias and Q/K resonance).
"""
import math

import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_helpers import F16_MODEL_FACTOR, f16_score_rmse_model, rel_errors
from oracle import pseudo_average as pa


def emulated_f16_attention(q, k, v, causal, mode, rows):
    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = k.shape
    g = Hq // Hkv
    scale = 1.0 / math.sqrt(D)
    kk, means = pa.kshift(k) if mode == 0 else (k, None)
    out = []
    for r in rows:
        b, rem = divmod(int(r), Hq * Sq)
        h, i = divmod(rem, Sq)
        hk = h // g
        lim = min(Sk, i + Sk - Sq + 1) if causal else Sk
        qi = q[b, h, i].astype(np.float64)
        kb = kk[b, hk, :lim].astype(np.float64)
        acc = np.zeros(lim, np.float16)
        for st in range(D // 16):
            part = kb[:, 16 * st:16 * st + 16] @ qi[16 * st:16 * st + 16]   # exact: 16 products of fp16 values
            acc = (acc.astype(np.float64) + part).astype(np.float16)        # one rounding per step
        s = acc.astype(np.float64)
        if means is not None:
            s = s + np.repeat(means[b, hk].astype(np.float64), pa.block_rows_for(D), axis=0)[:lim] @ qi
        s = scale * s
        p = np.exp(s - s.max())
        p /= p.sum()
        out.append(p @ v[b, hk, :lim].astype(np.float64))
    return np.array(out)


def _res(name, seed, freq):
    return wl.Workload(name, 1, 2, 2, 1024, 1024, 64, False, "resonance", seed,
                       (("A", 30.0), ("freq", freq), ("noise_std", 0.5), ("phase_flip", True)))


CASES = [
    _res("res_uniform", 5, "uniform_pi"),
    _res("res_rope", 6, "rope"),
    _res("res_slow", 7, "slow"),
    wl.Workload("kbias20", 1, 4, 2, 1024, 1024, 128, True, "kbias", 8, (("bias_std", 20.0),)),
    wl.Workload("kbias_t3", 1, 4, 2, 1024, 1024, 128, True, "kbias_t3", 9,
                (("bias_std", 10.0), ("t_dof", 3), ("t_scale", 4.0))),
    wl.Workload("iid", 1, 4, 2, 1024, 1024, 128, True, "iid", 10),
]


@pytest.mark.parametrize("mode", [0, 2], ids=["shift_f16acc", "naive_f16acc"])
@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_model_bounds_emulated_fp16_accumulation(w, mode):
    q, k, v = wl.make_inputs(w)
    rows = np.arange(0, w.B * w.Hq * w.Sq, 23)
    o_ref, _ = oracle.attention(q, k, v, causal=w.causal, rows=rows)
    err = rel_errors(emulated_f16_attention(q, k, v, w.causal, mode, rows), o_ref)[0]
    pred = f16_score_rmse_model(q, k, v, w.causal, mode, rows)
    print(f"\n{w.name} mode {mode}: emulated {err:.3e} predicted {pred:.3e} ratio {err / pred:.2f}")
    assert err <= F16_MODEL_FACTOR * pred, (err, pred)
    # not vacuous: within 4x, except where the raw resonance partial sums cancel (the naive
    # kernel on uniform frequencies), where the spacing at |S| overstates the partials' spacing
    if not (mode == 2 and w.name == "res_uniform"):
        assert pred <= 4.0 * err, (err, pred)
