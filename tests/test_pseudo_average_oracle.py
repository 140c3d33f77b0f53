"""Pins for the pseudo-average / shifted-key reference (oracle/pseudo_average.py).

The abstract of "Online Pseudo-average Shifting Attention (PASA) for Robust Low-precision
LLM Inference" (arXiv 2503.01873) names the step ("online pseudo-average shifting") but
does not define it; the reading is documented in the module. These tests pin that reading
by closed forms (constant blocks, exact means, rounding ties), bounds that any correct
implementation satisfies (on the grid, within one grid step of the true mean, never above
the block's largest magnitude), and the equivalence the abstract states: shifting and then
recovering gives plain attention.
"""
import numpy as np
import pytest

from oracle import pseudo_average as pa


def f16(x):
    return np.asarray(x, dtype=np.float64).astype(np.float16)


def test_grid_step_is_fp16_ulp():
    vals = f16([0.0, 2.0 ** -24, 2.0 ** -15, 2.0 ** -14, 1.0, 1.5, 2.0, 1000.0, 60000.0])
    got = pa.grid_step(vals)
    nxt = np.nextafter(vals, np.float16(np.inf)).astype(np.float64) - vals.astype(np.float64)
    np.testing.assert_array_equal(got, nxt)
    assert pa.grid_step(f16([65504.0]))[0] == 32.0


def test_constant_block_gives_constant_mean_and_zero_shift():
    for c in (0.0, 1.0, -3.25, 20.5, 1e-3, 60000.0 / 4):
        kb = f16(np.full((112, 8), c))
        m = pa.block_pseudo_average(kb)
        assert np.all(m == kb[0]), c


def test_exact_mean_on_grid():
    # values on the grid of the block maximum with an exactly representable mean
    kb = f16(np.array([[1.0, -2.0], [3.0, -2.0], [5.0, 4.0], [7.0, 4.0]]))
    m = pa.block_pseudo_average(kb)
    np.testing.assert_array_equal(m.astype(np.float64), [4.0, 1.0])


def test_round_half_even_ties():
    # n = 2 and an odd sum of grid units: the mean is exactly halfway between two grid
    # points and rounds to the even one. Channel maxima lie in [0.125, 0.25), grid 2^-13.
    u = 2.0 ** -13
    kb = f16(np.array([[2016 * u, 2016 * u, 2016 * u], [1985 * u, 1987 * u, 1986 * u]]))
    m = pa.block_pseudo_average(kb).astype(np.float64)
    assert m[0] == 2000 * u    # 2000.5 -> 2000
    assert m[1] == 2002 * u    # 2001.5 -> 2002
    assert m[2] == 2001 * u    # 2001 exactly
    # negative tie: -2000.5 -> -2000
    m = pa.block_pseudo_average(-kb).astype(np.float64)
    assert m[0] == -2000 * u and m[1] == -2002 * u


def test_bounds_on_random_blocks():
    rng = np.random.default_rng(0)
    for trial in range(50):
        n = int(rng.integers(1, 113))
        scale = 10.0 ** rng.uniform(-4, 3)
        bias = rng.normal(0, 20) * scale
        kb = f16(rng.standard_normal((n, 16)) * scale + bias)
        m = pa.block_pseudo_average(kb).astype(np.float64)
        x = kb.astype(np.float64)
        M = np.abs(x).max(0)
        g = pa.grid_step(f16(M))
        assert np.all(np.abs(m) <= M)
        assert np.all(np.mod(m, g) == 0), "the pseudo-average lies on the grid of the block maximum"
        # each element moves by at most g/2 when quantised, the mean by at most g/2 when rounded
        assert np.all(np.abs(m - x.mean(0)) <= g + 1e-300)


def test_tail_block_uses_valid_rows_only():
    rng = np.random.default_rng(1)
    k = f16(rng.standard_normal((1, 1, 250, 8)) * 3 + 5)
    ks, means = pa.kshift(k, block_rows=112)
    assert means.shape == (1, 1, 3, 8)
    np.testing.assert_array_equal(means[0, 0, 2], pa.block_pseudo_average(k[0, 0, 224:250]))
    ks2, means2 = pa.kshift_fast(k, block_rows=112)
    np.testing.assert_array_equal(means2, means)
    np.testing.assert_array_equal(ks2.view(np.uint16), ks.view(np.uint16))


def test_guard_for_huge_channels_and_nonfinite():
    kb = f16(np.array([[40000.0, 1.0, np.inf], [-30000.0, 3.0, 2.0]]))
    m = pa.block_pseudo_average(kb).astype(np.float64)
    assert m[0] == 0.0   # max |K| >= 2^15: no shift, so K - m cannot overflow
    assert m[1] == 2.0
    assert m[2] == 0.0   # inf in the block: no shift


def test_shift_is_mostly_exact_and_removes_bias():
    # the point of rounding the mean to the grid: K - m is exact in fp16 for most elements
    rng = np.random.default_rng(2)
    k = f16(rng.standard_normal((1, 2, 448, 64)) + rng.normal(0, 20, (1, 2, 1, 64)))
    ks, means = pa.kshift_fast(k, block_rows=112)
    exact = ks.astype(np.float64) == k.astype(np.float64) - np.repeat(means.astype(np.float64), 112, axis=2)
    assert exact.mean() > 0.85
    assert np.abs(ks.astype(np.float64)).max() < 8.0       # bias of ~20 per channel removed
    assert np.abs(k.astype(np.float64)).max() > 30.0


def test_shifted_value_is_correctly_rounded():
    # K' = fp16(K - m) with one rounding: compare against the two fp16 neighbours
    rng = np.random.default_rng(3)
    k = f16(rng.standard_normal((1, 1, 224, 32)) * rng.uniform(0.01, 100, 32))
    ks, means = pa.kshift_fast(k, block_rows=112)
    exact = k.astype(np.float64) - np.repeat(means.astype(np.float64), 112, axis=2)
    got = ks.astype(np.float64)
    lo = np.nextafter(ks, np.float16(-np.inf)).astype(np.float64)
    hi = np.nextafter(ks, np.float16(np.inf)).astype(np.float64)
    assert np.all(np.abs(got - exact) <= np.abs(lo - exact))
    assert np.all(np.abs(got - exact) <= np.abs(hi - exact))


@pytest.mark.parametrize("causal", [False, True])
def test_shift_then_recover_equals_plain_attention(oracle_mod, causal):
    # data on a coarse grid so every shifted value is exact: recovered == plain attention
    rng = np.random.default_rng(4)
    q = f16(rng.integers(-3, 4, (1, 4, 40, 16)))
    k = f16(rng.integers(-20, 21, (1, 2, 230, 16)) + rng.integers(-100, 100, (1, 2, 1, 16)))
    v = f16(rng.standard_normal((1, 2, 230, 16)))
    ks, means = pa.kshift(k, block_rows=112)
    exact = ks.astype(np.float64) == k.astype(np.float64) - np.repeat(means.astype(np.float64), 112, axis=2)[:, :, :230]
    assert exact.all()
    o0, l0 = oracle_mod.attention(q, k, v, causal=causal, scale=0.05)
    o1, l1 = oracle_mod.attention_recovered(q, ks, means, 112, v, causal=causal, scale=0.05)
    np.testing.assert_allclose(o1, o0, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l1, l0, rtol=1e-12, atol=1e-12)
    # and without the offsets the result is wrong: the recovery step is load-bearing
    o2, _ = oracle_mod.attention(q, ks, v, causal=causal, scale=0.05)
    assert np.abs(o2 - o0).max() > 1e-3


def test_recovered_score_magnitude_equals_raw_when_shift_is_exact(oracle_mod):
    # q . (k' + m) = q . k when k' = k - m exactly (coarse-grid data); the shifted magnitude
    # itself is much smaller because the per-channel bias is gone
    rng = np.random.default_rng(6)
    q = f16(rng.integers(-3, 4, (1, 4, 30, 16)))
    k = f16(rng.integers(-20, 21, (1, 2, 230, 16)) + rng.integers(-200, 200, (1, 2, 1, 16)))
    ks, means = pa.kshift(k, block_rows=112)
    for causal in (False, True):
        raw = oracle_mod.row_max_abs_score(q, k, causal)
        rec = oracle_mod.row_max_abs_recovered(q, ks, means, 112, causal)
        np.testing.assert_array_equal(rec, raw)
        assert np.median(raw / np.maximum(oracle_mod.row_max_abs_score(q, ks, causal), 1)) > 2


# ---------------------------------------------------------------------------------------
# The alternative reading kept as a switch: m = the exact block mean rounded once to fp16.


def test_fp16_round_rational_against_single_roundings():
    # num / den exactly representable in float64 (den a power of two): numpy's float64 ->
    # float16 conversion is then a single correct rounding to compare against
    rng = np.random.default_rng(11)
    for _ in range(3000):
        e = int(rng.integers(0, 40))
        num = int(rng.integers(-(1 << 40), 1 << 40)) >> int(rng.integers(0, 30))
        val = num / float(1 << e)
        if abs(val) >= 65504:
            continue
        assert pa.fp16_round_rational(num, 1 << e) == float(np.float16(val))
    # ties go to the even neighbour, in the normal and the subnormal range
    assert pa.fp16_round_rational(2049, 2) == 1024.0          # 1024.5: between 1024 and 1025
    assert pa.fp16_round_rational(2051, 2) == 1026.0          # 1025.5: between 1025 and 1026
    assert pa.fp16_round_rational(3, 1 << 25) == 2.0 ** -23   # 1.5 * 2^-24
    assert pa.fp16_round_rational(1, 1 << 25) == 0.0          # 0.5 * 2^-24
    assert pa.fp16_round_rational(1, 3) == float(np.float16(1 / 3))


def test_plain_rule_closed_forms():
    kb = f16([[1.0, 1024.0, 5.0, -7.0], [2.0, 1025.0, 5.0, -7.0]])
    m = pa.block_pseudo_average(kb, "plain").astype(np.float64)
    assert m[0] == 1.5          # exact mean, representable
    assert m[1] == 1024.0       # 1024.5 rounds to the even neighbour
    assert m[2] == 5.0 and m[3] == -7.0
    # where the exact mean is on the grid of the block maximum the two readings agree
    kb = f16(np.arange(-8, 8).reshape(16, 1) * np.ones((1, 3)))
    np.testing.assert_array_equal(pa.block_pseudo_average(kb, "plain"), pa.block_pseudo_average(kb, "grid"))
    # and they differ where the mean falls between grid points of the maximum: values
    # {1000, 0.25}: mean 500.125, grid of 1000 is 0.5 (-> 500.0), fp16 spacing at 500 is
    # 0.25 (-> 500.0 as well; a tie to even); {1000, 0.75}: mean 500.375 -> grid 500.5,
    # plain 500.5 (tie, even); {1000, 1.5}: mean 500.75 -> grid 501.0 (tie at 0.5 spacing
    # 500.5 / 501.0 -> even 501.0), plain 500.75
    kb = f16([[1000.0], [1.5]])
    assert float(pa.block_pseudo_average(kb, "grid")[0]) == 501.0
    assert float(pa.block_pseudo_average(kb, "plain")[0]) == 500.75


def test_plain_rule_guard_and_tail():
    kb = f16(np.array([[40000.0, 1.0, np.inf], [-30000.0, 3.0, 2.0]]))
    m = pa.block_pseudo_average(kb, "plain").astype(np.float64)
    assert m[0] == 0.0 and m[1] == 2.0 and m[2] == 0.0
    rng = np.random.default_rng(12)
    k = f16(rng.standard_normal((2, 2, 250, 8)) * 3 + 40)
    ks, means = pa.kshift(k, block_rows=112, rule="plain")
    for b in range(2):
        for h in range(2):
            for j, (r0, r1) in enumerate([(0, 112), (112, 224), (224, 250)]):
                ex = k[b, h, r0:r1].astype(np.float64).mean(axis=0)   # exact enough for the bound
                mj = means[b, h, j].astype(np.float64)
                spacing = np.abs(np.nextafter(means[b, h, j], np.float16(np.inf)).astype(np.float64) - mj)
                assert np.all(np.abs(mj - ex) <= spacing)


def test_plain_rule_fast_equals_exact():
    rng = np.random.default_rng(13)
    for scale, bias in [(1.0, 0.0), (3.0, 40.0), (1e-4, 0.0), (200.0, 3000.0)]:
        k = f16(rng.standard_normal((1, 3, 300, 16)) * scale + bias * rng.standard_normal((1, 3, 1, 16)))
        ks1, m1 = pa.kshift(k, block_rows=128, rule="plain")
        ks2, m2 = pa.kshift_fast(k, block_rows=128, rule="plain")
        np.testing.assert_array_equal(m1.view(np.uint16), m2.view(np.uint16))
        np.testing.assert_array_equal(ks1.view(np.uint16), ks2.view(np.uint16))


def test_grid_rule_keeps_more_shifted_keys_exact_than_plain():
    # the reason for the grid reading: K - m stays exact in fp16 where the plain mean has
    # bits below the keys' own spacing (a mean near zero: unbiased or resonance keys)
    rng = np.random.default_rng(14)
    t = np.arange(512)[None, None, :, None]
    cases = {
        "iid": rng.standard_normal((1, 4, 512, 64)),
        "resonance": 30 * np.sin(t * rng.uniform(0, np.pi, (1, 4, 1, 64)) + rng.uniform(0, 6.3, (1, 4, 1, 64)))
        + rng.normal(0, 0.5, (1, 4, 512, 64)),
        "bias20": rng.standard_normal((1, 4, 512, 64)) + rng.normal(0, 20, (1, 4, 1, 64)),
    }
    for name, x in cases.items():
        k = f16(x)
        frac = {}
        for rule in ("grid", "plain"):
            ks, means = pa.kshift_fast(k, block_rows=128, rule=rule)
            exact = ks.astype(np.float64) == k.astype(np.float64) - np.repeat(means.astype(np.float64), 128, axis=2)
            frac[rule] = exact.mean()
        assert frac["grid"] > 0.85, (name, frac)
        assert frac["grid"] >= frac["plain"], (name, frac)
        if name != "bias20":
            assert frac["plain"] < 0.5, (name, frac)


@pytest.mark.parametrize("causal", [False, True])
def test_plain_rule_shift_then_recover_equals_plain_attention(oracle_mod, causal):
    rng = np.random.default_rng(15)
    q = f16(rng.integers(-3, 4, (1, 4, 40, 16)))
    k = f16(rng.integers(-20, 21, (1, 2, 230, 16)) + rng.integers(-100, 100, (1, 2, 1, 16)))
    v = f16(rng.standard_normal((1, 2, 230, 16)))
    ks, means = pa.kshift(k, block_rows=112, rule="plain")
    o0, l0 = oracle_mod.attention(q, k, v, causal=causal, scale=0.05)
    o1, l1 = oracle_mod.attention_recovered(q, ks, means, 112, v, causal=causal, scale=0.05)
    # K - m may be inexact here (m off the integer grid): agreement to the fp16 rounding of K'
    np.testing.assert_allclose(o1, o0, rtol=0, atol=5e-3)
    np.testing.assert_allclose(l1, l0, rtol=0, atol=5e-3)
