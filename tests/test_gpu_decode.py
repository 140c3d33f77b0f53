"""GPU parity of the decode path: a few query rows per head against a key cache.

"Online Pseudo-average Shifting Attention (PASA) for Robust Low-precision LLM Inference"
(arXiv 2503.01873), Abstract: the method targets long-sequence inference. In decoding the
keys live in a cache; the pseudo-average of a key block depends on that block's rows
alone, so the shifted cache and its block means stay valid as rows are appended, and only
the block that an append touches is recomputed (pasa_kshift_blocks). pasa_attn_fwd_decode
packs the g query heads of a kv group into one tile and splits the key blocks across CTAs;
the split results are merged by their log-sum-exps (inside a thread-block cluster for up
to 8 splits at D = 128, else by a second kernel). The result must be attention up to
rounding: the same gates as the prefill parity tests, against the same fp64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_helpers import f16all_bound, lse_tolerance, rel_errors, to_dev

pytestmark = pytest.mark.gpu

MODES = [0, 1, 2, 3, 4]
MODE_NAMES = {0: "shift_f16acc", 1: "shift_f32acc", 2: "naive_f16acc", 3: "noshift_f32acc", 4: "shift_f16all"}
BN = 128   # key block rows (both head dims)


def pasa():
    import precision_flashattention_numerics_gb300 as p

    return p


def inputs(B, Hq, Hkv, Sq, Sk, D, kind, seed, **params):
    w = wl.Workload("decode", B, Hq, Hkv, Sq, Sk, D, False, kind, seed, tuple(sorted(params.items())))
    return wl.make_inputs(w)


def prepared(k, mode):
    """Device cache for `mode`: shifted keys and means (modes 0, 1, 4) or raw keys."""
    p = pasa()
    (kt,) = to_dev(k)
    if mode in (0, 1, 4):
        return p.kshift(kt)
    return kt, None


def decode(q, k, v, causal, mode, splits=0):
    p = pasa()
    qt, vt = to_dev(q, v)
    ks, means = prepared(k, mode)
    o, lse = p.attn_fwd_decode(qt, ks, means, vt, causal=causal, mode=mode, splits=splits)
    p.check_device_error()
    return o, lse


def gate(kind, mode):
    if mode == 2 and kind != "iid":
        return (5e-2, 2e-1)   # the naive fp16 kernel is only expected to stay finite here
    if kind != "iid":
        return (5e-3, 5e-2)
    return (2e-3, 1e-2)


CASES = [
    # (B, Hq, Hkv, Sq, Sk, D, causal, kind, params, splits)
    (1, 8, 1, 1, 5000, 128, False, "kbias", {"bias_std": 20.0}, 0),      # g = 8, one row per head
    (2, 28, 4, 4, 3001, 128, True, "kbias_t3", {"bias_std": 10.0, "t_dof": 3, "t_scale": 4.0}, 0),  # g = 7
    (1, 4, 4, 16, 1000, 64, True, "iid", {}, 3),
    (1, 16, 2, 8, 2049, 64, False, "iid", {}, 0),                       # 64 packed rows
    (1, 2, 1, 64, 777, 128, True, "iid", {}, 100),                      # 128 packed rows, a split per block
    (3, 6, 3, 1, 130, 128, True, "iid", {}, 0),                         # two blocks: unsplit
    (1, 4, 2, 2, 20000, 128, True, "kbias", {"bias_std": 20.0}, 0),
    (1, 8, 1, 1, 5000, 128, True, "kbias", {"bias_std": 20.0}, 12),     # > 8 splits: the merge kernel
    (2, 14, 2, 2, 3000, 128, True, "iid", {}, 8),                       # 8 splits: one cluster of 8
]


@pytest.mark.parametrize("mode", MODES, ids=[MODE_NAMES[m] for m in MODES])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_decode_parity(case, mode):
    B, Hq, Hkv, Sq, Sk, D, causal, kind, params, splits = CASES[case]
    q, k, v = inputs(B, Hq, Hkv, Sq, Sk, D, kind, 500 + case, **params)
    o, lse = decode(q, k, v, causal, mode, splits)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal)
    og = o.double().cpu().numpy()
    lg = lse.double().cpu().numpy()
    assert np.isfinite(og).all()
    if mode == 4:
        # the fp16 accumulation bound over all of the cache's blocks also covers a split,
        # whose fp16 accumulator sees fewer of them
        base = 5e-2 if kind != "iid" else 1e-2
        bound = base * np.abs(o_ref).max() + f16all_bound(Sk) * float(np.abs(v.astype(np.float64)).max())
        assert np.abs(og - o_ref).max() <= bound
    else:
        rmse, rmax = rel_errors(og, o_ref)
        tol = gate(kind, mode)
        assert rmse <= tol[0] and rmax <= tol[1], (rmse, rmax)
    fin = np.isfinite(lse_ref)
    assert np.all(np.isneginf(lg[~fin]))
    assert np.max(np.abs(lg[fin] - lse_ref[fin])) <= lse_tolerance(q, k, causal, mode, D)


@pytest.mark.parametrize("mode", MODES, ids=[MODE_NAMES[m] for m in MODES])
@pytest.mark.parametrize("g,Sq,D,causal", [(7, 16, 128, True), (8, 2, 64, True), (1, 1, 128, False),
                                           (4, 3, 128, True), (8, 4, 128, True)])
def test_single_split_against_the_prefill_kernel(g, Sq, D, causal, mode):
    """One split. More than 32 packed rows, or D = 64, run the attention kernel on the packed
    rows. Where pasa_attn_fwd_shifted runs that same kernel (D = 128, or the fp16-PV mode at
    D = 64) every row goes through the same per-row arithmetic, so O and LSE are
    bit-identical. Otherwise (the swapped-operand decode kernel for up to 32 rows at
    D = 128; the two-set prefill kernel at D = 64) the scores, offsets and row sums are the
    same numbers summed in another order, so O agrees to a few fp16 roundings of P
    (relative 2^-10 per term) and the LSE to fp32 rounding."""
    p = pasa()
    Hkv, Sk = 2, 1500
    q, k, v = inputs(2, g * Hkv, Hkv, Sq, Sk, D, "kbias", 40 + g, bias_std=10.0)
    qt, vt = to_dev(q, v)
    ks, means = prepared(k, mode)
    o1, l1 = p.attn_fwd_decode(qt, ks, means, vt, causal=causal, mode=mode, splits=1)
    o2, l2 = p.attn_fwd_shifted(qt, ks, means, vt, causal=causal, mode=mode)
    p.check_device_error()
    same_kernel = (D == 128 and g * Sq > 32) or (D == 64 and mode == 4)
    if same_kernel:
        assert torch.equal(o1, o2)
        assert torch.equal(l1, l2)
    else:
        d = (o1.double() - o2.double()).abs().max().item()
        scale = o2.double().abs().max().item()
        tol = f16all_bound(Sk) if mode == 4 else 2e-3
        assert d <= tol * scale, (d, scale)
        assert (l1.double() - l2.double()).abs().max().item() <= (f16all_bound(Sk) if mode == 4 else 1e-4)


def test_fp16_pv_decode_differs_from_fp32_pv():
    """Mode 4 keeps O and the row sums in fp16: on flat attention (iid keys, 5000 cached)
    its result must differ from mode 0 somewhere, and stay within the fp16 bound."""
    p = pasa()
    B, Hq, Hkv, Sq, Sk, D = 1, 8, 2, 1, 5000, 128
    q, k, v = inputs(B, Hq, Hkv, Sq, Sk, D, "iid", 4242)
    o0, _ = decode(q, k, v, True, 0)
    o4, _ = decode(q, k, v, True, 4)
    o_ref, _ = oracle.attention(q, k, v, causal=True)
    assert not torch.equal(o0, o4)
    d4 = np.abs(o4.double().cpu().numpy() - o_ref).max()
    assert d4 <= 1e-2 * np.abs(o_ref).max() + f16all_bound(Sk) * float(np.abs(v.astype(np.float64)).max())


@pytest.mark.parametrize("mode", [0, 3])
def test_cache_rows_past_the_length_are_not_read(mode):
    """A cache of cap rows holding Sk valid ones: rows past Sk (here NaN, and means blocks
    past the last one, also NaN) must not reach the result, which equals the dense call."""
    p = pasa()
    B, Hq, Hkv, Sq, Sk, cap, D = 2, 8, 2, 2, 1300, 2000, 128
    q, k, v = inputs(B, Hq, Hkv, Sq, Sk, D, "kbias", 77, bias_std=20.0)
    qt, kt, vt = to_dev(q, k, v)
    nan = float("nan")
    kc = torch.full((B, Hkv, cap, D), nan, device="cuda", dtype=torch.float16)
    vc = torch.full((B, Hkv, cap, D), nan, device="cuda", dtype=torch.float16)
    kc[:, :, :Sk] = kt
    vc[:, :, :Sk] = vt
    nbc = -(-cap // BN)
    ksc = torch.full_like(kc, nan)
    mc = torch.full((B, Hkv, nbc, D), nan, device="cuda", dtype=torch.float16)
    if mode == 0:
        p.kshift_blocks(kc, ksc, mc, 0, length=Sk)
        ks, means = p.kshift(kt)
        nb = -(-Sk // BN)
        assert torch.equal(ksc[:, :, :Sk], ks) and torch.equal(mc[:, :, :nb], means)
        assert torch.isnan(ksc[:, :, Sk:]).all() and torch.isnan(mc[:, :, nb:]).all()
    else:
        ksc, mc, ks, means = kc, None, kt, None
    for splits in (0, 1, 4):
        o1, l1 = p.attn_fwd_decode(qt, ksc, mc, vc, causal=True, mode=mode, splits=splits, length=Sk)
        o2, l2 = p.attn_fwd_decode(qt, ks, means, vt, causal=True, mode=mode, splits=splits)
        p.check_device_error()
        assert torch.isfinite(o1).all()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("D", [64, 128])
def test_kshift_blocks_after_append(D):
    """Shift a cache of 300 rows, append 250 and refresh from the block the append touched
    (block 2, which held 44 rows): every row and mean equals a full pasa_kshift of the 550
    rows, and nothing past them is written."""
    p = pasa()
    B, H, cap, S0, S1 = 2, 3, 1000, 300, 550
    _, k, _ = inputs(B, H, H, 1, cap, D, "kbias", 9, bias_std=20.0)
    (kc,) = to_dev(k)
    sentinel = 1234.0
    ksc = torch.full_like(kc, sentinel)
    mc = torch.full((B, H, -(-cap // BN), D), sentinel, device="cuda", dtype=torch.float16)
    p.kshift_blocks(kc, ksc, mc, 0, length=S0)
    ks0, m0 = p.kshift(kc[:, :, :S0].contiguous())
    assert torch.equal(ksc[:, :, :S0], ks0) and torch.equal(mc[:, :, :3], m0)
    assert (ksc[:, :, S0:] == sentinel).all() and (mc[:, :, 3:] == sentinel).all()
    p.kshift_blocks(kc, ksc, mc, S0 // BN, length=S1)
    ks1, m1 = p.kshift(kc[:, :, :S1].contiguous())
    p.check_device_error()
    assert torch.equal(ksc[:, :, :S1], ks1) and torch.equal(mc[:, :, :5], m1)
    assert (ksc[:, :, S1:] == sentinel).all() and (mc[:, :, 5:] == sentinel).all()


def test_decode_loop_against_the_oracle():
    """Prefill 250 keys, then 6 decode steps of one query row per head, each appending its
    key/value row to the cache, refreshing the touched block and attending causally."""
    p = pasa()
    B, Hq, Hkv, D, S0, steps, cap = 1, 8, 2, 128, 250, 6, 512
    q, k, v = inputs(B, Hq, Hkv, steps, S0 + steps, D, "kbias", 123, bias_std=20.0)
    (kt, vt) = to_dev(k, v)
    kc = torch.zeros((B, Hkv, cap, D), device="cuda", dtype=torch.float16)
    vc = torch.zeros_like(kc)
    ksc = torch.zeros_like(kc)
    mc = torch.zeros((B, Hkv, cap // BN, D), device="cuda", dtype=torch.float16)
    kc[:, :, :S0], vc[:, :, :S0] = kt[:, :, :S0], vt[:, :, :S0]
    p.kshift_blocks(kc, ksc, mc, 0, length=S0)
    for t in range(steps):
        Sk = S0 + t + 1
        kc[:, :, Sk - 1], vc[:, :, Sk - 1] = kt[:, :, Sk - 1], vt[:, :, Sk - 1]
        p.kshift_blocks(kc, ksc, mc, (Sk - 1) // BN, length=Sk)
        qs = np.ascontiguousarray(q[:, :, t:t + 1])
        (qt,) = to_dev(qs)
        o, lse = p.attn_fwd_decode(qt, ksc, mc, vc, causal=True, mode=0, length=Sk)
        p.check_device_error()
        o_ref, lse_ref = oracle.attention(qs, k[:, :, :Sk], v[:, :, :Sk], causal=True)
        rmse, rmax = rel_errors(o.double().cpu().numpy(), o_ref)
        assert rmse <= 5e-3 and rmax <= 5e-2, (t, rmse, rmax)
        assert np.abs(lse.double().cpu().numpy() - lse_ref).max() <= lse_tolerance(qs, k[:, :, :Sk], True, 0, D)


def test_full_size_decode():
    """The decode workload at full cache length (Qwen2-7B-like heads: Hq = 28, Hkv = 4,
    D = 128; 32768 cached keys with a heavy-tailed sequence-dimension bias), B = 2 here to
    bound host memory; automatic split, compared row by row with the oracle. Gates as in
    the prefill full-size tests: relRMSE <= 5e-3 on biased keys for modes 0, 1, 3; the naive
    fp16 mode and the fp16-PV mode are reported and must stay finite."""
    B, Hq, Hkv, Sq, Sk, D = 2, 28, 4, 1, 32768, 128
    q, k, v = inputs(B, Hq, Hkv, Sq, Sk, D, "kbias_t3", 2024, bias_std=10.0, t_dof=3, t_scale=4.0)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=True)
    for mode in (0, 1, 2, 3, 4):
        o, lse = decode(q, k, v, True, mode)
        og = o.double().cpu().numpy()
        rmse, rmax = rel_errors(og, o_ref)
        print(f"\nfull-size decode, mode {mode}: relRMSE={rmse:.3e} relMax={rmax:.3e}")
        assert np.isfinite(og).all()
        if mode in (2, 4):
            continue   # as in the prefill full-size tests: reported only on biased heavy-tailed keys
        assert rmse <= 5e-3, (mode, rmse, rmax)
        assert np.abs(lse.double().cpu().numpy() - lse_ref).max() <= lse_tolerance(q, k, True, mode, D)


STEP_CASES = [
    # (B, Hq, Hkv, Sq, Sk, cap, D, splits): the swapped-operand kernel with the in-cluster
    # merge, one split, the workspace merge (> 8 splits), 32 packed rows, and the attention
    # kernel on packed rows (D = 64; 48 rows)
    (2, 28, 4, 1, 5000, 5120, 128, 0),
    (1, 8, 2, 2, 1100, 1280, 128, 1),
    (1, 4, 1, 1, 9000, 9216, 128, 12),
    (2, 16, 2, 4, 3000, 3072, 128, 0),
    (1, 8, 2, 1, 2000, 2048, 64, 0),
    (1, 24, 2, 4, 700, 768, 128, 0),
]


@pytest.mark.parametrize("mode", [0, 1, 4, 2])
@pytest.mark.parametrize("case", range(len(STEP_CASES)))
def test_decode_step_equals_refresh_then_decode(case, mode):
    """pasa_attn_fwd_decode_step after an append (the last block rewritten in the raw cache)
    gives the shifted cache, the means, O and the LSE of pasa_kshift_blocks followed by
    pasa_attn_fwd_decode, bit for bit; its decode kernel overlaps the refresh and waits for
    it only before the refreshed blocks."""
    p = pasa()
    B, Hq, Hkv, Sq, Sk, cap, D, splits = STEP_CASES[case]
    q, k, v = inputs(B, Hq, Hkv, Sq, cap, D, "kbias_t3", 300 + case, bias_std=10.0, t_dof=3, t_scale=4.0)
    qt, kt, vt = to_dev(q, k, v)
    nbc = -(-cap // BN)
    first = (Sk - Sq) // BN   # the block the Sq appended rows start in
    caches = []
    for _ in range(2):
        ks = torch.zeros_like(kt)
        m = torch.zeros((B, Hkv, nbc, D), device="cuda", dtype=torch.float16)
        p.kshift_blocks(kt, ks, m, 0, length=Sk - Sq)   # the cache before the append
        caches.append((ks, m))
    (ka, ma), (kb, mb) = caches
    shift = mode in (0, 1, 4)
    if shift:
        p.kshift_blocks(kt, ka, ma, first, length=Sk)
    o_a, l_a = p.attn_fwd_decode(qt, ka if shift else kt, ma if shift else None, vt, causal=True, mode=mode,
                                 splits=splits, length=Sk)
    o_b, l_b = p.attn_fwd_decode_step(qt, kt, kb if shift else kt, mb if shift else None, vt, first, causal=True,
                                      mode=mode, splits=splits, length=Sk)
    torch.cuda.synchronize()
    p.check_device_error()
    assert torch.equal(o_a, o_b) and torch.equal(l_a, l_b)
    if shift:
        assert torch.equal(ka, kb) and torch.equal(ma, mb)


def test_decode_step_loop_against_the_oracle():
    """Decode steps through pasa_attn_fwd_decode_step, each appending one key/value row per
    head: checked against the fp64 oracle at every step."""
    p = pasa()
    B, Hq, Hkv, D, S0, steps, cap = 2, 28, 4, 128, 4090, 8, 4224
    q, k, v = inputs(B, Hq, Hkv, steps, S0 + steps, D, "kbias", 124, bias_std=20.0)
    (kt, vt) = to_dev(k, v)
    kc = torch.zeros((B, Hkv, cap, D), device="cuda", dtype=torch.float16)
    vc = torch.zeros_like(kc)
    ksc = torch.zeros_like(kc)
    mc = torch.zeros((B, Hkv, cap // BN, D), device="cuda", dtype=torch.float16)
    kc[:, :, :S0], vc[:, :, :S0] = kt[:, :, :S0], vt[:, :, :S0]
    p.kshift_blocks(kc, ksc, mc, 0, length=S0)
    for t in range(steps):
        Sk = S0 + t + 1
        kc[:, :, Sk - 1], vc[:, :, Sk - 1] = kt[:, :, Sk - 1], vt[:, :, Sk - 1]
        qs = np.ascontiguousarray(q[:, :, t:t + 1])
        (qt,) = to_dev(qs)
        o, lse = p.attn_fwd_decode_step(qt, kc, ksc, mc, vc, (Sk - 1) // BN, causal=True, mode=0, length=Sk)
        p.check_device_error()
        o_ref, lse_ref = oracle.attention(qs, k[:, :, :Sk], v[:, :, :Sk], causal=True)
        rmse, rmax = rel_errors(o.double().cpu().numpy(), o_ref)
        assert rmse <= 5e-3 and rmax <= 5e-2, (t, rmse, rmax)
        assert np.abs(lse.double().cpu().numpy() - lse_ref).max() <= lse_tolerance(qs, k[:, :, :Sk], True, 0, D)


def test_decode_step_and_one_call_prefill_on_a_side_stream():
    """The calls that launch a kernel with programmatic dependence on the key preparation
    (the decode step; the one-call prefill) give the same results on a non-default stream
    as the separate calls on the default one, with work queued on that stream around them."""
    p = pasa()
    B, Hq, Hkv, Sq, Sk, cap, D = 2, 28, 4, 1, 3000, 3072, 128
    q, k, v = inputs(B, Hq, Hkv, Sq, cap, D, "kbias", 77, bias_std=20.0)
    qt, kt, vt = to_dev(q, k, v)
    first = (Sk - 1) // BN
    ka, ma = torch.zeros_like(kt), torch.zeros((B, Hkv, cap // BN, D), device="cuda", dtype=torch.float16)
    p.kshift_blocks(kt, ka, ma, 0, length=Sk)
    o_a, l_a = p.attn_fwd_decode(qt, ka, ma, vt, causal=True, mode=0, length=Sk)
    qp, kp, vp = to_dev(*inputs(1, 8, 2, 700, 700, D, "kbias", 78, bias_std=10.0))
    ks, means = p.kshift(kp)
    o_pa, l_pa = p.attn_fwd_shifted(qp, ks, means, vp, causal=True, mode=0)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        kb, mb = torch.zeros_like(kt), torch.zeros_like(ma)
        p.kshift_blocks(kt, kb, mb, 0, length=Sk - 1)
        o_b, l_b = p.attn_fwd_decode_step(qt, kt, kb, mb, vt, first, causal=True, mode=0, length=Sk)
        o_pb, l_pb = p.attn_fwd(qp, kp, vp, causal=True, mode=0)
        o_b2 = o_b.clone()   # stream-ordered after the step
    side.synchronize()
    p.check_device_error()
    assert torch.equal(o_a, o_b) and torch.equal(l_a, l_b) and torch.equal(o_b2, o_a)
    assert torch.equal(ka, kb) and torch.equal(ma, mb)
    assert torch.equal(o_pa, o_pb) and torch.equal(l_pa, l_pb)
