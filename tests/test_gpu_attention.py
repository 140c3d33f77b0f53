"""GPU parity of the attention forward pass against the fp64 oracle.

"Online Pseudo-average Shifting Attention (PASA) for Robust Low-precision LLM Inference"
(arXiv 2503.01873), Abstract: PASA is mathematically equivalent to plain attention, keeps
fp16 scores from overflowing (65504) under large sequence-dimension bias and Q/K
resonance, and is evaluated by RMSE against high-precision attention. Tolerances (output
scale): relRMSE <= 2e-3 and relMax <= 1e-2 on unbiased data; no inf/NaN and relRMSE <= 5e-3
on biased and resonance data, except where the scores are accumulated in fp16 at
magnitudes where that cannot hold (resonance keys: shifted scores near 1e4, fp16 spacing
8-16): there the gate is 2x the relRMSE that an fp16 accumulator's rounding predicts
(gpu_helpers.f16_score_rmse_model). LSE is compared in absolute terms.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_helpers import (f16_score_rmse_gate, f16_score_rmse_model, f16all_bound, gather_rows, lse_tolerance,
                         rel_errors, to_dev)

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
MODES = [0, 1, 2, 3]
MODE_NAMES = {0: "shift_f16acc", 1: "shift_f32acc", 2: "naive_f16acc", 3: "noshift_f32acc", 4: "shift_f16all"}


def pasa():
    import precision_flashattention_numerics_gb300 as p

    return p


def run(q, k, v, causal, mode, scale=None):
    p = pasa()
    qt, kt, vt = to_dev(q, k, v)
    o, lse = p.attn_fwd(qt, kt, vt, causal=causal, scale=scale, mode=mode)
    p.check_device_error()
    return o, lse


def small_case(B, Hq, Hkv, Sq, Sk, D, kind, seed, **params):
    w = wl.Workload("small", B, Hq, Hkv, Sq, Sk, D, False, kind, seed, tuple(sorted(params.items())))
    return wl.make_inputs(w)


SMALL = [
    # (B, Hq, Hkv, Sq, Sk, D, causal, kind, params)
    (1, 2, 1, 300, 300, 64, False, "iid", {}),
    (1, 2, 1, 300, 300, 64, True, "iid", {}),
    (2, 4, 2, 520, 520, 128, True, "iid", {}),
    (1, 4, 2, 520, 520, 128, True, "kbias", {"bias_std": 20.0}),
    (1, 2, 2, 200, 333, 128, True, "iid", {}),      # Sk > Sq: bottom-right aligned mask
    (1, 2, 2, 333, 200, 64, True, "iid", {}),       # Sq > Sk: leading rows see no key
    (1, 1, 1, 64, 50, 64, False, "iid", {}),        # a single partial key block
    (1, 4, 1, 1, 500, 128, True, "iid", {}),        # one query row
    (1, 2, 2, 257, 1000, 128, False, "kbias_t3", {"bias_std": 10.0, "t_dof": 3, "t_scale": 4.0}),
]


@pytest.mark.parametrize("mode", MODES, ids=[MODE_NAMES[m] for m in MODES])
@pytest.mark.parametrize("case", range(len(SMALL)))
def test_small_parity(case, mode):
    B, Hq, Hkv, Sq, Sk, D, causal, kind, params = SMALL[case]
    q, k, v = small_case(B, Hq, Hkv, Sq, Sk, D, kind, 100 + case, **params)
    o, lse = run(q, k, v, causal, mode)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal)
    og = o.double().cpu().numpy()
    lg = lse.double().cpu().numpy()
    assert np.isfinite(og).all()
    rmse, rmax = rel_errors(og, o_ref)
    biased = kind != "iid"
    if mode == 2 and biased:
        tol = (5e-2, 2e-1)   # the naive fp16 kernel is only expected to stay finite here
    elif biased:
        tol = (5e-3, 5e-2)
    else:
        tol = (2e-3, 1e-2)
    assert rmse <= tol[0] and rmax <= tol[1], (rmse, rmax)
    fin = np.isfinite(lse_ref)
    assert np.all(np.isneginf(lg[~fin]))
    assert np.all(og.reshape(-1, D)[~fin.reshape(-1)] == 0.0)
    assert np.max(np.abs(lg[fin] - lse_ref[fin])) <= lse_tolerance(q, k, causal, mode, D)


@pytest.mark.parametrize("causal", [False, True])
def test_hand_worked_example(causal):
    # tests/golden/hand_example.json, zero-padded from D = 2 to D = 64 (same scores)
    ex = json.load(open(os.path.join(HERE, "golden", "hand_example.json")))
    def pad(x):
        a = np.zeros(np.array(x).shape[:-1] + (64,))
        a[..., :2] = np.array(x)
        return a.astype(np.float16)
    q, k, v = pad(ex["q"]), pad(ex["k"]), pad(ex["v"])
    ref = ex["causal" if causal else "noncausal"]
    for mode in MODES:
        o, lse = run(q, k, v, causal, mode, scale=ex["scale"])
        og = o.double().cpu().numpy()[..., :2]
        np.testing.assert_allclose(og, np.array(ref["o"]), rtol=0, atol=1e-2 * 14)
        assert np.all(o.double().cpu().numpy()[..., 2:] == 0)
        np.testing.assert_allclose(lse.double().cpu().numpy(), np.log(np.array(ref["lse_exp"], float)),
                                   atol=2e-3)


@pytest.mark.parametrize("mode", MODES, ids=[MODE_NAMES[m] for m in MODES])
def test_invariants(mode):
    p = pasa()
    rng = np.random.default_rng(11)
    B, Hq, Hkv, S, D = 1, 4, 2, 400, 128
    q = (rng.standard_normal((B, Hq, S, D))).astype(np.float16)
    k = (rng.standard_normal((B, Hkv, S, D))).astype(np.float16)
    v = (rng.standard_normal((B, Hkv, S, D))).astype(np.float16)
    ones = np.ones_like(v)
    # rows of P sum to one: V = 1 gives O = 1 (fp16 rounding of P only)
    o, _ = run(q, k, ones, True, mode)
    assert np.abs(o.double().cpu().numpy() - 1.0).max() <= 2e-3
    # causal row 0 sees key 0 only: O_0 = V_0 exactly
    o, _ = run(q, k, v, True, mode)
    og = o.cpu().numpy()
    for h in range(Hq):
        np.testing.assert_array_equal(og[0, h, 0], v[0, h // 2, 0])
    # a single key: O = V_0 exactly, LSE = scale q . k_0
    o1, l1 = run(q, k[:, :, :1].copy(), v[:, :, :1].copy(), False, mode)
    og1 = o1.cpu().numpy()
    for h in range(Hq):
        np.testing.assert_array_equal(og1[0, h], np.broadcast_to(v[0, h // 2, 0], (S, D)))
    lref = (q.astype(np.float64) @ np.repeat(k[:, :, :1], 2, axis=1).astype(np.float64).transpose(0, 1, 3, 2))[..., 0]
    assert np.abs(l1.double().cpu().numpy() - lref / math.sqrt(D)).max() <= 1e-2
    # GQA equals MHA with the key/value heads repeated, bit for bit
    kr = np.ascontiguousarray(np.repeat(k, 2, axis=1))
    vr = np.ascontiguousarray(np.repeat(v, 2, axis=1))
    o2, l2 = run(q, kr, vr, True, mode)
    assert torch.equal(o, o2)


def test_f32acc_shift_matches_noshift_on_unbiased_data():
    rng = np.random.default_rng(12)
    q = rng.standard_normal((1, 2, 700, 128)).astype(np.float16)
    k = rng.standard_normal((1, 2, 700, 128)).astype(np.float16)
    v = rng.standard_normal((1, 2, 700, 128)).astype(np.float16)
    o1, _ = run(q, k, v, False, 1)
    o3, _ = run(q, k, v, False, 3)
    rmse, rmax = rel_errors(o1.double().cpu().numpy(), o3.double().cpu().numpy())
    assert rmse < 1e-3 and rmax < 1e-2


def test_recovered_reference_isolates_accumulation_error():
    # Using the kernel's own shifted keys and means, the fp64 "shift then recover" reference
    # matches plain attention closely and the GPU output matches both.
    p = pasa()
    q, k, v = small_case(1, 4, 2, 520, 520, 128, "kbias", 5, bias_std=20.0)
    (kt,) = to_dev(k)
    ks, means = p.kshift(kt)
    ks, means = ks.cpu().numpy(), means.cpu().numpy()
    o_rec, _ = oracle.attention_recovered(q, ks, means, p.block_rows(128), v, causal=True)
    o_ref, _ = oracle.attention(q, k, v, causal=True)
    assert rel_errors(o_rec, o_ref)[0] < 1e-3
    o, _ = run(q, k, v, True, 1)
    assert rel_errors(o.double().cpu().numpy(), o_rec)[0] < 2e-3


# ---------------------------------------------------------------------------------------
# the measured workloads at full size, compared on sampled rows
# ---------------------------------------------------------------------------------------
FULL = wl.MEASURED + ["resonance_rope_a30_b2h5_s9216_d64", "resonance_slow_a30_b2h5_s9216_d64",
                      "resonance_hot_a48_b2h5_s9216_d64"]
_inputs_cache = {}


def full_inputs(name):
    if name not in _inputs_cache:
        _inputs_cache.clear()
        w = wl.WORKLOADS[name]
        q, k, v = wl.make_inputs(w)
        rows = wl.sample_rows(w, 160)
        o_ref, lse_ref = oracle.attention(q, k, v, causal=w.causal, rows=rows)
        _inputs_cache[name] = (w, (q, k, v), to_dev(q, k, v), rows, o_ref, lse_ref)
    return _inputs_cache[name]


# (relRMSE, relMax) gates per (workload, mode). The fp16-accumulated score modes on biased
# and resonance inputs, and mode 4 everywhere, are gated on the fp16-accumulation error
# model of gpu_helpers.f16_score_rmse_model (a relRMSE bound, no relMax): on resonance keys
# the shifted scores stay near 1e4 (fp16 spacing 8-16), where no fixed 5e-3 holds for an
# fp16 accumulator, but a kernel that loses accuracy beyond its accumulator still fails.
_model_cache = {}


def gate(name, w, mode):
    unbiased = w.kind == "iid"
    if mode in (0, 2, 4) and (not unbiased or mode == 4):
        if (name, mode) not in _model_cache:
            _, (q, k, v), _, rows, _, _ = full_inputs(name)
            _model_cache[(name, mode)] = f16_score_rmse_model(q, k, v, w.causal, mode, rows)
        pred = _model_cache[(name, mode)]
        g = f16_score_rmse_gate(pred)
        if mode == 0 and w.kind != "resonance":
            g = min(g, 5e-3)    # PASA on biased keys also keeps the contract's 5e-3
        return g, None, pred
    return ((2e-3, 1e-2) if unbiased else (5e-3, None)) + (None,)


FULL_CASES = [(n, m) for n in FULL for m in MODES + [4]]


@pytest.mark.parametrize("name,mode", FULL_CASES, ids=[f"{n}-{MODE_NAMES[m]}" for n, m in FULL_CASES])
def test_full_size_sampled_rows(name, mode):
    p = pasa()
    w, host, (qt, kt, vt), rows, o_ref, lse_ref = full_inputs(name)
    o, lse = p.attn_fwd(qt, kt, vt, causal=w.causal, mode=mode)
    p.check_device_error()
    n_bad = int((~torch.isfinite(o)).sum().item())
    og = gather_rows(o, rows)
    lg = lse.reshape(-1)[torch.as_tensor(rows, device=o.device)].double().cpu().numpy()
    rmse, rmax = rel_errors(og, o_ref) if n_bad == 0 else (float("nan"), float("nan"))
    print(f"\n{name} mode={MODE_NAMES[mode]} nonfinite={n_bad} relRMSE={rmse:.3e} relMax={rmax:.3e} "
          f"lse_maxerr={np.nanmax(np.abs(lg - lse_ref)):.3e}")
    if name.startswith("resonance_hot") and mode == 2:
        assert n_bad > 0, "the naive fp16 kernel is expected to overflow on this input"
        return
    assert n_bad == 0
    g_rmse, g_rmax, pred = gate(name, w, mode)
    if pred is not None:
        print(f"fp16-score model: predicted relRMSE {pred:.3e}, gate {g_rmse:.3e}, measured/predicted "
              f"{rmse / pred:.2f}")
    assert rmse <= g_rmse, (rmse, g_rmse)
    if g_rmax is not None:
        assert rmax <= g_rmax, (rmax, g_rmax)


# ---------------------------------------------------------------------------------------
# mode 4: half precision throughout the loop (fp16 PV accumulator, fp16 running row sum)
# ---------------------------------------------------------------------------------------
@pytest.mark.parametrize("case", range(len(SMALL)))
def test_f16all_small_parity(case):
    B, Hq, Hkv, Sq, Sk, D, causal, kind, params = SMALL[case]
    q, k, v = small_case(B, Hq, Hkv, Sq, Sk, D, kind, 100 + case, **params)
    o, lse = run(q, k, v, causal, 4)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal)
    og = o.double().cpu().numpy()
    lg = lse.double().cpu().numpy()
    assert np.isfinite(og).all()
    # the mode-0 part of the error (relative to max |O|, as gated in test_small_parity) plus
    # the fp16 accumulation bound, elementwise
    base = 5e-2 if kind != "iid" else 1e-2
    bound = base * np.abs(o_ref).max() + f16all_bound(Sk) * float(np.abs(v.astype(np.float64)).max())
    assert np.abs(og - o_ref).max() <= bound, (np.abs(og - o_ref).max(), bound)
    rmse, rmax = rel_errors(og, o_ref)
    print(f"\nf16all case {case}: relRMSE={rmse:.3e} relMax={rmax:.3e} bound/max|O|={bound / np.abs(o_ref).max():.3e}")
    fin = np.isfinite(lse_ref)
    assert np.all(np.isneginf(lg[~fin]))
    assert np.max(np.abs(lg[fin] - lse_ref[fin])) <= lse_tolerance(q, k, causal, 4, D)


def moving_max_case(seed=31, S=1000, D=128):
    """Scores that rise by about 100 (12.75 in the kernel's log2 units, more than its lazy
    threshold of 8) from each 128-key block to the next, so the running max moves at every
    block and the O rescale runs each time. Channel 0 carries the rise: q[0] = 25 and
    k[0] = 4 * block index (constant within a block, so the pseudo-average takes it whole and
    the offsets q . m_j carry it)."""
    rng = np.random.default_rng(seed)
    q = 0.5 * rng.standard_normal((1, 2, S, D))
    k = 0.5 * rng.standard_normal((1, 2, S, D))
    v = rng.standard_normal((1, 2, S, D))
    q[..., 0] = 25.0
    k[..., 0] = 4.0 * (np.arange(S) // 128)[None, None, :]
    return q.astype(np.float16), k.astype(np.float16), v.astype(np.float16)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4], ids=[MODE_NAMES[m] for m in range(5)])
def test_running_max_moves(mode, causal):
    q, k, v = moving_max_case()
    D = q.shape[-1]
    o, lse = run(q, k, v, causal, mode)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal)
    og = o.double().cpu().numpy()
    lg = lse.double().cpu().numpy()
    assert np.isfinite(og).all()
    rmse, rmax = rel_errors(og, o_ref)
    if mode == 4:
        bound = 5e-2 * np.abs(o_ref).max() + f16all_bound(k.shape[2]) * float(np.abs(v.astype(np.float64)).max())
        assert np.abs(og - o_ref).max() <= bound
    elif mode == 2:
        # raw scores up to ~800 accumulated in fp16 (spacing 0.5): the naive kernel gets the
        # same gate as on the other large-score inputs of test_small_parity
        assert rmse <= 5e-2 and rmax <= 2e-1, (rmse, rmax)
    else:
        assert rmse <= 5e-3 and rmax <= 5e-2, (rmse, rmax)
    assert np.max(np.abs(lg - lse_ref)) <= lse_tolerance(q, k, causal, mode, D)


def test_f16all_differs_from_f32_accumulation():
    # mode 4 really accumulates PV in fp16: on 1000 keys its output is not bit-identical to
    # mode 0's, while both stay within their bounds of the oracle (tests above)
    q, k, v = moving_max_case(seed=32)
    o0, _ = run(q, k, v, False, 0)
    o4, _ = run(q, k, v, False, 4)
    assert not torch.equal(o0, o4)


# ---------------------------------------------------------------------------------------
# pasa_attn_fwd itself (the contract's signature: the library takes its shift workspace
# from the stream-ordered allocator), called through ctypes and compared with the oracle
# ---------------------------------------------------------------------------------------
def _attn_fwd_c_abi(q, k, v, causal, mode):
    import ctypes

    lib = pasa().library()
    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = k.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Sq), device=q.device, dtype=torch.float32)
    P = ctypes.c_void_p
    rc = lib.pasa_attn_fwd(P(q.data_ptr()), P(k.data_ptr()), P(v.data_ptr()), P(o.data_ptr()), P(lse.data_ptr()),
                           B, Hq, Hkv, Sq, Sk, D, int(causal), 0.0, mode, P(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, lib.pasa_strerror(rc)
    pasa().check_device_error()
    return o, lse


C_ABI_CASES = [
    # (B, Hq, Hkv, Sq, Sk, D, causal, kind, params): K bias 20 non-causal; causal GQA with a ragged tail
    (1, 4, 4, 640, 700, 128, False, "kbias", {"bias_std": 20.0}),
    (2, 6, 2, 333, 333, 64, True, "iid", {}),
    (1, 8, 2, 1000, 1000, 128, True, "kbias_t3", {"bias_std": 10.0, "t_dof": 3, "t_scale": 4.0}),
]


@pytest.mark.parametrize("mode", [0, 1], ids=[MODE_NAMES[m] for m in (0, 1)])
@pytest.mark.parametrize("case", range(len(C_ABI_CASES)))
def test_pasa_attn_fwd_c_abi_against_oracle(case, mode):
    B, Hq, Hkv, Sq, Sk, D, causal, kind, params = C_ABI_CASES[case]
    q, k, v = small_case(B, Hq, Hkv, Sq, Sk, D, kind, 400 + case, **params)
    qt, kt, vt = to_dev(q, k, v)
    o, lse = _attn_fwd_c_abi(qt, kt, vt, causal, mode)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal)
    og = o.double().cpu().numpy()
    lg = lse.double().cpu().numpy()
    assert np.isfinite(og).all()
    rmse, rmax = rel_errors(og, o_ref)
    tol = (5e-3, 5e-2) if kind != "iid" else (2e-3, 1e-2)
    assert rmse <= tol[0] and rmax <= tol[1], (rmse, rmax)
    fin = np.isfinite(lse_ref)
    assert np.all(np.isneginf(lg[~fin]))
    assert np.max(np.abs(lg[fin] - lse_ref[fin])) <= lse_tolerance(q, k, causal, mode, D)
    # and the same bytes as the workspace entry point the other tests use
    o_ws, lse_ws = pasa().attn_fwd(qt, kt, vt, causal=causal, mode=mode)
    assert torch.equal(o, o_ws) and torch.equal(lse, lse_ws)


# ---------------------------------------------------------------------------------------
# seeded random sweep: shapes, ragged lengths, GQA ratios, masks, modes and both key paths
# (pre-pass and fused shift), each against the oracle with the gates used above
# ---------------------------------------------------------------------------------------
def _sweep_cases(n=32, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for t in range(n):
        D = int(rng.choice([64, 128]))
        Hkv = int(rng.integers(1, 4))
        g = int(rng.choice([1, 2, 4, 7]))
        Sq = int(rng.integers(1, 700))
        Sk = int(max(1, Sq + rng.integers(-300, 400)))
        causal = bool(rng.integers(0, 2))
        kind = str(rng.choice(["iid", "kbias", "kbias_t3"]))
        mode = int(rng.choice([0, 1, 2, 3, 4]))
        fused = D == 128 and mode in (0, 1, 4) and bool(rng.integers(0, 2))
        out.append((int(rng.integers(1, 3)), Hkv * g, Hkv, Sq, Sk, D, causal, kind, mode, fused, 700 + t))
    return out


SWEEP = _sweep_cases()


@pytest.mark.parametrize("case", SWEEP, ids=[f"{c[5]}d-{c[1]}/{c[2]}h-{c[3]}x{c[4]}-{'c' if c[6] else 'n'}-{c[7]}-m{c[8]}"
                                             f"{'-fused' if c[9] else ''}" for c in SWEEP])
def test_random_sweep_against_oracle(case):
    B, Hq, Hkv, Sq, Sk, D, causal, kind, mode, fused, seed = case
    params = {"iid": {}, "kbias": {"bias_std": 20.0}, "kbias_t3": {"bias_std": 10.0, "t_dof": 3, "t_scale": 4.0}}[kind]
    q, k, v = small_case(B, Hq, Hkv, Sq, Sk, D, kind, seed, **params)
    p = pasa()
    qt, kt, vt = to_dev(q, k, v)
    if fused:
        o, lse = p.attn_fwd_fused(qt, kt, vt, causal=causal, mode=mode)
    else:
        o, lse = p.attn_fwd(qt, kt, vt, causal=causal, mode=mode)
    p.check_device_error()
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal)
    og = o.double().cpu().numpy()
    lg = lse.double().cpu().numpy()
    assert np.isfinite(og).all()
    fin = np.isfinite(lse_ref)
    assert np.all(np.isneginf(lg[~fin])) and np.all(og.reshape(-1, D)[~fin.reshape(-1)] == 0.0)
    if not fin.any():
        return
    rmse, rmax = rel_errors(og.reshape(-1, D)[fin.reshape(-1)], o_ref.reshape(-1, D)[fin.reshape(-1)])
    if mode == 4:
        bound = (5e-2 if kind != "iid" else 1e-2) * np.abs(o_ref).max() + f16all_bound(Sk) * float(
            np.abs(v.astype(np.float64)).max())
        assert np.abs(og - o_ref).max() <= bound
    elif mode == 2 and kind != "iid":
        assert rmse <= 5e-2 and rmax <= 2e-1, (rmse, rmax)
    elif kind != "iid":
        assert rmse <= 5e-3 and rmax <= 5e-2, (rmse, rmax)
    else:
        assert rmse <= 2e-3 and rmax <= 1e-2, (rmse, rmax)
    assert np.max(np.abs(lg[fin] - lse_ref[fin])) <= lse_tolerance(q, k, causal, mode, D)


@pytest.mark.parametrize("D,mode", [(128, 0), (128, 1), (128, 4), (128, 5), (64, 0), (64, 1)])
def test_back_to_back_calls_share_a_workspace(D, mode):
    """pasa_attn_fwd_ws launches the key preparation and then the attention kernel, which may
    start before the preparation ends and waits for it (griddepcontrol) before reading the
    prepared keys. Three calls on different inputs, queued without a host synchronisation
    on one workspace, must each equal the preparation and the attention run as separate
    calls on their own buffers, bit for bit: no call may read another's prepared keys."""
    p = pasa()
    B, Hq, Hkv, S = 1, 8, 2, 1500
    ins = [to_dev(*wl.make_inputs(wl.Workload("ws", B, Hq, Hkv, S, S, D, True, "kbias", 900 + i,
                                              (("bias_std", 10.0),)))) for i in range(3)]
    ws = torch.empty(p.library().pasa_attn_fwd_workspace_bytes(B, Hkv, S, D, mode), device="cuda",
                     dtype=torch.uint8)
    outs = [p.attn_fwd(q, k, v, causal=True, mode=mode, workspace=ws) for (q, k, v) in ins]
    torch.cuda.synchronize()
    p.check_device_error()
    for (q, k, v), (o, lse) in zip(ins, outs):
        if mode == 5:
            k8, means, kscale = p.kprep_fp8(k, mode=mode)
            o_ref, lse_ref = p.attn_fwd_fp8(q, k8, means, kscale, v, causal=True, mode=mode)
        else:
            ks, means = p.kshift(k)
            o_ref, lse_ref = p.attn_fwd_shifted(q, ks, means, v, causal=True, mode=mode)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
