"""GPU: the pseudo-average shift kernel is bit-exact with the numpy reference.

PASA Abstract ("online pseudo-average shifting"): the block means and the shifted keys are
integer-exact quantities under the reading in oracle/pseudo_average.py, so the CUDA result
must match the reference bit for bit.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_helpers import to_dev
from oracle import pseudo_average as pa

pytestmark = pytest.mark.gpu


def run(k):
    import precision_flashattention_numerics_gb300 as pasa

    (kt,) = to_dev(k)
    ks, means = pasa.kshift(kt)
    pasa.check_device_error()
    return ks.cpu().numpy(), means.cpu().numpy()


def f16(x):
    return np.asarray(x, dtype=np.float64).astype(np.float16)


@pytest.mark.parametrize("B,H,Sk,D,kind", [
    (1, 2, 300, 64, "iid"),
    (1, 1, 1, 64, "iid"),
    (1, 1, 128, 128, "iid"),    # exactly one block (128 keys)
    (1, 1, 129, 128, "iid"),    # one key past it
    (1, 1, 128, 64, "iid"),
    (1, 1, 129, 64, "iid"),
    (1, 4, 4096, 128, "kbias"),
    (2, 3, 1000, 128, "kbias_t3"),
    (2, 5, 9216, 64, "resonance"),
])
def test_kshift_bit_exact(B, H, Sk, D, kind):
    params = {"iid": (), "kbias": (("bias_std", 20.0),),
              "kbias_t3": (("bias_std", 10.0), ("t_dof", 3), ("t_scale", 4.0)),
              "resonance": (("A", 30.0), ("freq", "uniform_pi"), ("noise_std", 0.5), ("phase_flip", True))}[kind]
    w = wl.Workload("t", B, H, H, 16, Sk, D, False, kind, 77 + Sk, params)
    _, k, _ = wl.make_inputs(w)
    ks_ref, m_ref = pa.kshift_fast(k)
    ks, m = run(k)
    np.testing.assert_array_equal(m.view(np.uint16), m_ref.view(np.uint16))
    np.testing.assert_array_equal(ks.view(np.uint16), ks_ref.view(np.uint16))


def test_kshift_special_values():
    rng = np.random.default_rng(5)
    k = rng.standard_normal((1, 2, 250, 64)) * 3 + 7
    k[0, 0, 5, 3] = np.inf                 # channel with inf: no shift
    k[0, 0, 120:200, 4] = 40000.0          # |K| >= 2^15: no shift
    k[0, 0, 120:130, 5] = -60000.0
    k[0, 1, :, 6] = 0.0                    # all zeros
    k[0, 1, :, 7] = 2.0 ** -20             # subnormal fp16 values
    k[0, 1, 7, 8] = 6e-8
    k[0, 1, 224:, 9] = 65504.0             # tail block at the top of the range
    k = f16(k)
    ks_ref, m_ref = pa.kshift_fast(k)
    ks, m = run(k)
    np.testing.assert_array_equal(m.view(np.uint16), m_ref.view(np.uint16))
    np.testing.assert_array_equal(ks.view(np.uint16), ks_ref.view(np.uint16))
    assert m[0, 0, 0, 3] == 0 and np.isinf(ks[0, 0, 5, 3])


# ---------------------------------------------------------------------------------------
# The plain fp16-rounded block mean (pasa_kshift_mean, PASA_MEAN_PLAIN) against the oracle's
# exact rational rounding of the same reading.

def run_plain(k):
    import precision_flashattention_numerics_gb300 as pasa

    (kt,) = to_dev(k)
    ks, means = pasa.kshift(kt, mean_rule=pasa.MEAN_PLAIN)
    pasa.check_device_error()
    return ks.cpu().numpy(), means.cpu().numpy()


@pytest.mark.parametrize("B,H,Sk,D,kind", [
    (1, 2, 300, 64, "iid"),
    (1, 1, 1, 64, "iid"),
    (1, 1, 129, 128, "iid"),
    (1, 4, 4096, 128, "kbias"),
    (2, 3, 1000, 128, "kbias_t3"),
    (2, 5, 2000, 64, "resonance"),
])
def test_kshift_plain_mean_bit_exact(B, H, Sk, D, kind):
    params = {"iid": (), "kbias": (("bias_std", 20.0),),
              "kbias_t3": (("bias_std", 10.0), ("t_dof", 3), ("t_scale", 4.0)),
              "resonance": (("A", 30.0), ("freq", "uniform_pi"), ("noise_std", 0.5), ("phase_flip", True))}[kind]
    w = wl.Workload("t", B, H, H, 16, Sk, D, False, kind, 91 + Sk, params)
    _, k, _ = wl.make_inputs(w)
    ks_ref, m_ref = pa.kshift(k, rule="plain") if B * H * Sk <= 4000 else pa.kshift_fast(k, rule="plain")
    ks, m = run_plain(k)
    np.testing.assert_array_equal(m.view(np.uint16), m_ref.view(np.uint16))
    np.testing.assert_array_equal(ks.view(np.uint16), ks_ref.view(np.uint16))


def test_kshift_plain_mean_special_values_and_ties():
    rng = np.random.default_rng(6)
    k = rng.standard_normal((1, 2, 250, 64)) * 3 + 7
    k[0, 0, 5, 3] = np.inf
    k[0, 0, 120:200, 4] = 40000.0
    k[0, 1, :, 6] = 0.0
    k[0, 1, :, 7] = 2.0 ** -20
    k[0, 1, 7, 8] = 6e-8
    k[0, 1, 224:, 9] = 65504.0
    k[0, 0, :128, 10] = 1024.0             # block 0, channel 10: mean 1024.5, a tie -> 1024
    k[0, 0, :64, 10] = 1025.0
    k[0, 0, :128, 11] = 2.0 ** -24         # mean 1.5 * 2^-24: a subnormal tie -> 2^-23
    k[0, 0, :64, 11] = 2.0 ** -23
    k = f16(k)
    ks_ref, m_ref = pa.kshift(k, rule="plain")
    ks, m = run_plain(k)
    np.testing.assert_array_equal(m.view(np.uint16), m_ref.view(np.uint16))
    np.testing.assert_array_equal(ks.view(np.uint16), ks_ref.view(np.uint16))
    assert float(m[0, 0, 0, 10]) == 1024.0 and float(m[0, 0, 0, 11]) == 2.0 ** -23


def test_mean_rules_accuracy():
    """Modes 0 and 1 on K' from each rule (pasa_attn_fwd_shifted), against the fp64 oracle.
    Both are attention up to rounding. In the fp16-score mode the score accumulation
    dominates either way; in the fp32-score mode the rounding of K' is what is left, and
    the grid reading, which keeps K - m exact far more often, loses less where the mean is
    small against the block maximum (resonance keys)."""
    import oracle
    import precision_flashattention_numerics_gb300 as pasa
    from gpu_helpers import rel_errors

    cases = [("kbias", 4, 2, 1000, 128, (("bias_std", 20.0),)),
             ("iid", 4, 2, 1000, 128, ()),
             ("resonance", 2, 2, 1500, 64, (("A", 30.0), ("freq", "uniform_pi"), ("noise_std", 0.5),
                                            ("phase_flip", True)))]
    for kind, Hq, Hkv, S, D, params in cases:
        w = wl.Workload("t", 1, Hq, Hkv, S, S, D, kind != "resonance", kind, 303, params)
        q, k, v = wl.make_inputs(w)
        o_ref, _ = oracle.attention(q, k, v, causal=w.causal)
        qt, kt, vt = to_dev(q, k, v)
        for mode in (pasa.MODE_SHIFT_F16ACC, pasa.MODE_SHIFT_F32ACC):
            errs = {}
            for rule in (pasa.MEAN_GRID, pasa.MEAN_PLAIN):
                ks, means = pasa.kshift(kt, mean_rule=rule)
                o, _ = pasa.attn_fwd_shifted(qt, ks, means, vt, causal=w.causal, mode=mode)
                pasa.check_device_error()
                og = o.double().cpu().numpy()
                assert np.isfinite(og).all()
                errs[rule] = rel_errors(og, o_ref)
            print(f"\n{kind} mode {mode}: grid relRMSE={errs[0][0]:.3e} relMax={errs[0][1]:.3e}; "
                  f"plain relRMSE={errs[1][0]:.3e} relMax={errs[1][1]:.3e}")
            if kind != "resonance" or mode == pasa.MODE_SHIFT_F32ACC:
                assert errs[0][0] <= 5e-3 and errs[1][0] <= 5e-3
            if kind == "resonance" and mode == pasa.MODE_SHIFT_F32ACC:
                assert errs[0][0] <= errs[1][0]
