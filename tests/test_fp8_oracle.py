"""Pins of the oracle's e4m3 quantiser (oracle/fp8.py) against torch's float8_e4m3fn and the
format definition; see the module docstring for the reading of the scales."""
import numpy as np
import pytest
import torch

from oracle import fp8


def all_e4m3_values():
    """Every finite e4m3 value, decoded from the bit fields (sign, 4-bit exponent, 3-bit mantissa)."""
    vals = []
    for bits in range(256):
        s, e, m = bits >> 7, (bits >> 3) & 15, bits & 7
        if e == 15 and m == 7:
            continue                          # NaN
        v = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        vals.append(-v if s else v)
    return np.unique(np.array(vals))


def test_representable_values_are_fixed_points():
    v = all_e4m3_values()
    assert v.max() == 448.0 and np.min(v[v > 0]) == 2.0 ** -9
    np.testing.assert_array_equal(fp8.e4m3_round(v), v)


def test_midpoints_round_to_even_and_saturate():
    v = all_e4m3_values()
    pos = v[v >= 0]
    mids = (pos[:-1] + pos[1:]) / 2
    got = fp8.e4m3_round(mids)
    # a tie goes to the neighbour whose last mantissa bit is 0
    lo, hi = pos[:-1], pos[1:]
    even_lo = np.array([int(round(x / 2.0 ** (max(np.floor(np.log2(x)), -6) - 3))) % 2 == 0 if x > 0 else True
                        for x in lo])
    np.testing.assert_array_equal(got, np.where(even_lo, lo, hi))
    assert fp8.e4m3_round(np.array([500.0, -1e6]))[0] == 448.0
    assert fp8.e4m3_round(np.array([-1e6]))[0] == -448.0


def test_matches_torch_float8_e4m3fn_in_range():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(20000) * 10 ** rng.uniform(-4, 2.6, 20000),
                        all_e4m3_values()]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(fp8.e4m3_round(x.astype(np.float64)), want)


def test_row_and_block_scales():
    rng = np.random.default_rng(4)
    q = (rng.standard_normal((1, 2, 5, 16)) * 7).astype(np.float16)
    q8, sq = fp8.quantize_rows(q)
    # each row's largest magnitude maps to the largest code
    assert np.all(np.abs(q8).max(axis=-1) == 448.0)
    deq = q8 * sq.astype(np.float64)[..., None]
    # quantisation error at most half a spacing of the row's scale (3 mantissa bits: <= 1/16 relative)
    assert np.all(np.abs(deq - q.astype(np.float64)) <= np.abs(q.astype(np.float64)) / 16 + sq[..., None] * 2.0 ** -9)
    k = (rng.standard_normal((1, 1, 300, 16)) + 20).astype(np.float16)
    k8, sk = fp8.quantize_blocks(k, 128)
    assert sk.shape == (1, 1, 3)
    np.testing.assert_allclose(sk[0, 0, 2], np.float32(np.abs(k[0, 0, 256:].astype(np.float32)).max()) / np.float32(448))
    assert np.all(fp8.quantize_rows(np.zeros((1, 1, 2, 8), np.float16))[1] == 1.0)


def test_attention_fp8_reduces_to_plain_attention_on_e4m3_inputs(oracle_mod):
    # inputs whose rows / blocks are already e4m3 values with absmax 448 quantise exactly,
    # so the FP8 reference equals the plain fp64 oracle
    rng = np.random.default_rng(5)
    vals = all_e4m3_values()
    vals = vals[np.abs(vals) <= 8]
    q = rng.choice(vals, (1, 2, 40, 16)).astype(np.float16)
    k = rng.choice(vals, (1, 1, 200, 16)).astype(np.float16)
    q[..., 0] = 448.0
    k[..., 0, 0] = 448.0
    k[..., 128, 0] = 448.0
    v = rng.standard_normal((1, 1, 200, 16)).astype(np.float16)
    for causal in (False, True):
        o1, l1 = fp8.attention_fp8(q, k, v, causal, scale=0.01)
        o0, l0 = oracle_mod.attention(q, k, v, causal=causal, scale=0.01)
        np.testing.assert_allclose(o1, o0, rtol=1e-10, atol=1e-10)
        np.testing.assert_allclose(l1, l0, rtol=1e-10, atol=1e-10)
