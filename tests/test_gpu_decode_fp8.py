"""GPU: decode on an FP8 key cache (modes 5 and 6) against the oracle's e4m3 reading.

"Online Pseudo-average Shifting Attention (PASA) for Robust Low-precision LLM Inference"
(arXiv 2503.01873), Abstract: the shift keeps low-precision scores usable under a large
sequence-dimension bias of K; the method targets long-sequence inference. Here the cache
holds e4m3 codes of K' (mode 5) or K (mode 6) with one scale per 128-key block, refreshed
block-wise after an append (pasa_kprep_fp8_blocks), and the decode kernel quantises the new
query rows the same way the prefill FP8 kernel does. The gates are those of the prefill
FP8 parity tests: relRMSE <= 2e-3, relMax <= 1e-2 against fp64 attention on the
dequantised e4m3 values (oracle/fp8.py), LSE within 2e-3.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_helpers import rel_errors, to_dev
from oracle import fp8
from oracle import pseudo_average as pa

pytestmark = pytest.mark.gpu
BN = 128


def pasa():
    import precision_flashattention_numerics_gb300 as p

    return p


def inputs(B, Hq, Hkv, Sq, Sk, kind, seed, **params):
    w = wl.Workload("decf8", B, Hq, Hkv, Sq, Sk, 128, False, kind, seed, tuple(sorted(params.items())))
    return wl.make_inputs(w)


def oracle_fp8(q, k, v, causal, mode):
    if mode == 5:
        ks, means = pa.kshift_fast(k)
        return fp8.attention_fp8(q, ks, v, causal, means=means)
    return fp8.attention_fp8(q, k, v, causal)


def decode_fp8(q, k, v, causal, mode, splits=0):
    p = pasa()
    qt, kt, vt = to_dev(q, k, v)
    k8, means, kscale = p.kprep_fp8(kt, mode=mode)
    o, lse = p.attn_fwd_decode_fp8(qt, k8, means, kscale, vt, causal=causal, mode=mode, splits=splits)
    p.check_device_error()
    return o, lse


CASES = [
    # (B, Hq, Hkv, Sq, Sk, causal, kind, params, splits)
    (1, 8, 1, 1, 5000, False, "kbias", {"bias_std": 20.0}, 0),       # cluster merge (5 splits)
    (2, 28, 4, 4, 3001, True, "kbias_t3", {"bias_std": 10.0, "t_dof": 3, "t_scale": 4.0}, 0),  # 28 rows
    (1, 8, 2, 2, 2049, True, "iid", {}, 12),                          # the merge kernel
    (2, 6, 3, 1, 130, True, "iid", {}, 0),                            # one split
]


@pytest.mark.parametrize("mode", [5, 6])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_decode_fp8_matches_oracle_e4m3_reading(case, mode):
    B, Hq, Hkv, Sq, Sk, causal, kind, params, splits = CASES[case]
    q, k, v = inputs(B, Hq, Hkv, Sq, Sk, kind, 700 + case, **params)
    o, lse = decode_fp8(q, k, v, causal, mode, splits)
    o_ref, lse_ref = oracle_fp8(q, k, v, causal, mode)
    og = o.double().cpu().numpy()
    lg = lse.double().cpu().numpy()
    assert np.isfinite(og).all()
    rmse, rmax = rel_errors(og, o_ref)
    assert rmse <= 2e-3 and rmax <= 1e-2, (rmse, rmax)
    fin = np.isfinite(lse_ref)
    assert np.all(np.isneginf(lg[~fin]))
    assert np.max(np.abs(lg[fin] - lse_ref[fin])) <= 2e-3


@pytest.mark.parametrize("mode", [5, 6])
def test_decode_fp8_agrees_with_the_prefill_fp8_kernel(mode):
    """One split: the same e4m3 codes and scales as pasa_attn_fwd_fp8; the offsets (CUDA
    cores here, the tensor core there) and the row sums differ only in rounding order."""
    p = pasa()
    q, k, v = inputs(2, 8, 2, 2, 1500, "kbias", 41, bias_std=10.0)
    qt, kt, vt = to_dev(q, k, v)
    k8, means, kscale = p.kprep_fp8(kt, mode=mode)
    o1, l1 = p.attn_fwd_decode_fp8(qt, k8, means, kscale, vt, causal=True, mode=mode, splits=1)
    o2, l2 = p.attn_fwd_fp8(qt, k8, means, kscale, vt, causal=True, mode=mode)
    p.check_device_error()
    d = (o1.double() - o2.double()).abs().max().item()
    assert d <= 2e-3 * o2.double().abs().max().item(), d
    assert (l1.double() - l2.double()).abs().max().item() <= 1e-4


@pytest.mark.parametrize("mode", [5, 6])
def test_kprep_fp8_blocks_after_append(mode):
    """Prepare a cache of 300 rows, append 250 and refresh from the block the append touched:
    codes, block scales and means equal a full pasa_kprep_fp8 of the 550 rows, and nothing
    past them is written."""
    p = pasa()
    B, H, cap, S0, S1 = 2, 3, 1000, 300, 550
    _, k, _ = inputs(B, H, H, 1, cap, "kbias", 19, bias_std=20.0)
    (kc,) = to_dev(k)
    nbc = -(-cap // BN)
    k8 = torch.full((B, H, cap, 128), 0xAB, device="cuda", dtype=torch.uint8)
    ks = torch.full((B, H, nbc), -7.0, device="cuda", dtype=torch.float32)
    mc = torch.full((B, H, nbc, 128), 1234.0, device="cuda", dtype=torch.float16) if mode == 5 else None
    p.kprep_fp8_blocks(kc, k8, mc, ks, 0, mode=mode, length=S0)
    p.kprep_fp8_blocks(kc, k8, mc, ks, S0 // BN, mode=mode, length=S1)
    r8, rm, rs = p.kprep_fp8(kc[:, :, :S1].contiguous(), mode=mode)
    p.check_device_error()
    assert torch.equal(k8[:, :, :S1], r8) and torch.equal(ks[:, :, :5], rs)
    assert (k8[:, :, S1:] == 0xAB).all() and (ks[:, :, 5:] == -7.0).all()
    if mode == 5:
        assert torch.equal(mc[:, :, :5], rm) and (mc[:, :, 5:] == 1234.0).all()


@pytest.mark.parametrize("mode", [5, 6])
def test_decode_fp8_cache_rows_past_the_length_are_not_read(mode):
    p = pasa()
    B, Hq, Hkv, Sq, Sk, cap = 2, 8, 2, 2, 1300, 2000
    q, k, v = inputs(B, Hq, Hkv, Sq, Sk, "kbias", 79, bias_std=20.0)
    qt, kt, vt = to_dev(q, k, v)
    nan = float("nan")
    kc = torch.zeros((B, Hkv, cap, 128), device="cuda", dtype=torch.float16)
    vc = torch.full((B, Hkv, cap, 128), nan, device="cuda", dtype=torch.float16)
    kc[:, :, :Sk] = kt
    vc[:, :, :Sk] = vt
    nbc = -(-cap // BN)
    k8 = torch.full((B, Hkv, cap, 128), 0x7F, device="cuda", dtype=torch.uint8)   # e4m3 NaN past Sk
    ks = torch.full((B, Hkv, nbc), nan, device="cuda", dtype=torch.float32)
    mc = torch.full((B, Hkv, nbc, 128), nan, device="cuda", dtype=torch.float16) if mode == 5 else None
    p.kprep_fp8_blocks(kc, k8, mc, ks, 0, mode=mode, length=Sk)
    d8, dm, ds = p.kprep_fp8(kt, mode=mode)
    for splits in (0, 1, 4, 12):
        o1, l1 = p.attn_fwd_decode_fp8(qt, k8, mc, ks, vc, causal=True, mode=mode, splits=splits, length=Sk)
        o2, l2 = p.attn_fwd_decode_fp8(qt, d8, dm, ds, vt, causal=True, mode=mode, splits=splits)
        p.check_device_error()
        assert torch.isfinite(o1).all()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_shift_makes_fp8_decode_usable_on_biased_keys():
    """Against plain attention (fp64 oracle): e4m3 codes of the shifted keys keep their 3
    mantissa bits for the varying part of K; codes of the raw keys spend them on the bias."""
    q, k, v = inputs(1, 8, 2, 1, 4096, "kbias", 612, bias_std=20.0)
    o_ref, _ = oracle.attention(q, k, v, causal=True)
    err = {}
    for mode in (5, 6):
        o, _ = decode_fp8(q, k, v, True, mode)
        err[mode] = rel_errors(o.double().cpu().numpy(), o_ref)[0]
    print(f"\ndecode relRMSE vs plain attention: FP8 PASA {err[5]:.3e}, FP8 naive {err[6]:.3e}")
    assert err[5] < err[6] / 3, err


STEP_CASES = [
    # (B, Hq, Hkv, Sq, Sk, cap, splits): cluster merge, one split, the workspace merge, 32 rows
    (2, 28, 4, 1, 5000, 5120, 0),
    (1, 8, 2, 2, 1100, 1280, 1),
    (1, 4, 1, 1, 9000, 9216, 12),
    (2, 16, 2, 4, 3000, 3072, 0),
]


@pytest.mark.parametrize("mode", [5, 6])
@pytest.mark.parametrize("case", range(len(STEP_CASES)))
def test_decode_step_fp8_equals_refresh_then_decode(case, mode):
    """pasa_attn_fwd_decode_step_fp8 after an append gives the codes, block scales, means, O
    and LSE of pasa_kprep_fp8_blocks followed by pasa_attn_fwd_decode_fp8, bit for bit."""
    p = pasa()
    B, Hq, Hkv, Sq, Sk, cap, splits = STEP_CASES[case]
    q, k, v = inputs(B, Hq, Hkv, Sq, cap, "kbias_t3", 400 + case, bias_std=10.0, t_dof=3, t_scale=4.0)
    qt, kt, vt = to_dev(q, k, v)
    nbc = -(-cap // BN)
    first = (Sk - Sq) // BN
    caches = []
    for _ in range(2):
        k8 = torch.zeros((B, Hkv, cap, 128), device="cuda", dtype=torch.uint8)
        ks = torch.zeros((B, Hkv, nbc), device="cuda", dtype=torch.float32)
        mc = torch.zeros((B, Hkv, nbc, 128), device="cuda", dtype=torch.float16) if mode == 5 else None
        p.kprep_fp8_blocks(kt, k8, mc, ks, 0, mode=mode, length=Sk - Sq)   # before the append
        caches.append((k8, mc, ks))
    (k8a, ma, sa), (k8b, mb, sb) = caches
    p.kprep_fp8_blocks(kt, k8a, ma, sa, first, mode=mode, length=Sk)
    o_a, l_a = p.attn_fwd_decode_fp8(qt, k8a, ma, sa, vt, causal=True, mode=mode, splits=splits, length=Sk)
    o_b, l_b = p.attn_fwd_decode_step_fp8(qt, kt, k8b, mb, sb, vt, first, causal=True, mode=mode, splits=splits,
                                          length=Sk)
    torch.cuda.synchronize()
    p.check_device_error()
    assert torch.equal(o_a, o_b) and torch.equal(l_a, l_b)
    assert torch.equal(k8a, k8b) and torch.equal(sa, sb)
    if mode == 5:
        assert torch.equal(ma, mb)
