"""GPU: the FMA-pipe exponential the softmax runs on part of each key block's scores.

The attention kernels compute 2^x for 5 of every 16 score pairs with a Cody-Waite range
reduction and a fitted cubic (exp2_fma2) instead of MUFU ex2.approx, to balance the two
pipes. Its stated bound: relative error <= 7.5e-5 wherever the result is a normal fp32
number, a value in [0, 2^-125] for x <= -126 (masked scores are -inf), NaN in, NaN out.
Checked through the C ABI (pasa_selftest_exp2) against numpy's exp2 in fp64 and against the
MUFU outputs, on a dense sweep of the range the softmax uses (x <= 8 after the running max
is subtracted, down to the underflow) and on the special values.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

BOUND = 7.5e-5 * (1 + 1e-3)   # the fitted cubic's max relative error (fp32 Horner), with slack for rounding


def _run(x):
    import precision_flashattention_numerics_gb300 as p

    xt = torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()
    poly, mufu = p.selftest_exp2(xt)
    p.check_device_error()
    return poly.cpu().numpy().astype(np.float64), mufu.cpu().numpy().astype(np.float64)


def test_fma_exp2_relative_error_bound():
    rng = np.random.default_rng(3)
    # every fp32 step near 0 and the half-integers (where the reduction switches n), a
    # dense grid, and random values over [-125, 8]
    x = np.concatenate([np.linspace(-125.0, 8.0, 1_000_001), rng.uniform(-125.0, 8.0, 1_000_000),
                        np.arange(-125, 9) + 0.5, np.arange(-125, 9).astype(np.float64),
                        np.nextafter(np.float32(np.arange(-125, 9) + 0.5), np.float32(-1e9)),
                        np.nextafter(np.float32(np.arange(-125, 9) + 0.5), np.float32(1e9))]).astype(np.float32)
    poly, mufu = _run(x)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(poly - ref) / ref
    assert rel.max() <= BOUND, (rel.max(), x[np.argmax(rel)])
    # the MUFU exponential the other pairs use is far more accurate; both agree within the bound
    assert (np.abs(mufu - ref) / ref).max() <= 1e-6
    assert (np.abs(poly - mufu) / mufu).max() <= BOUND + 1e-6


def test_fma_exp2_underflow_and_special_values():
    x = np.array([-126.0, -126.4, -126.5, -127.0, -150.0, -1e4, -1e30, -np.inf, np.nan, np.inf, 0.0, -0.0, 8.0,
                  127.0], np.float32)
    poly, _ = _run(x)
    low = poly[:8]
    assert np.all((low >= 0.0) & (low <= 2.0 ** -125)), low           # 0 once rounded to fp16
    assert np.all(low.astype(np.float16) == 0)
    assert np.isnan(poly[8]) and not np.isfinite(poly[9])                # NaN in, NaN out; +inf not finite
    np.testing.assert_allclose(poly[10:], np.exp2(x[10:].astype(np.float64)), rtol=BOUND)
