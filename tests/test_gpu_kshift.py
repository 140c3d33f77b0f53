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
