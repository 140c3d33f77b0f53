"""GPU tests of pasa_attn_fwd_host: the PASA forward pass ("Online Pseudo-average Shifting
Attention (PASA) for Robust Low-precision LLM Inference", Abstract) on host buffers, staged
to the device in pieces (runs of (batch, kv head) units, or query-row ranges of one unit)
with the copies overlapped.

Each piece meets the same key blocks and pseudo-averages tile for tile, so the host-buffer
call must agree BIT FOR BIT with pasa_attn_fwd on device copies of the same inputs, for
every mode, piece plan and memory kind (pinned or pageable). One small case is also
checked against the fp64 oracle directly, with the bounds of the attention parity tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_helpers import lse_tolerance, rel_errors, to_dev

pytestmark = pytest.mark.gpu


def pasa():
    import precision_flashattention_numerics_gb300 as p

    return p


def make(B, Hq, Hkv, Sq, Sk, D, kind, seed, **params):
    w = wl.Workload("host", B, Hq, Hkv, Sq, Sk, D, False, kind, seed, tuple(sorted(params.items())))
    return wl.make_inputs(w)


def host_tensors(q, k, v, pinned=True):
    ts = [torch.from_numpy(np.ascontiguousarray(x)) for x in (q, k, v)]
    return [t.pin_memory() for t in ts] if pinned else ts


def device_result(q, k, v, causal, mode):
    p = pasa()
    qt, kt, vt = to_dev(q, k, v)
    o, lse = p.attn_fwd_alloc(qt, kt, vt, causal=causal, mode=mode)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


CASES = [
    # (B, Hq, Hkv, Sq, Sk, D, causal, kind, params)
    (2, 8, 4, 520, 520, 128, True, "iid", {}),
    (3, 6, 3, 300, 700, 64, True, "kbias", {"bias_std": 20.0}),
    (1, 4, 4, 257, 1000, 128, False, "kbias_t3", {"bias_std": 10.0, "t_dof": 3, "t_scale": 4.0}),
    (4, 8, 2, 1, 900, 128, True, "iid", {}),      # one query row per head
]


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4, 5, 6])
def test_host_matches_device(case, mode):
    B, Hq, Hkv, Sq, Sk, D, causal, kind, params = CASES[case]
    if mode >= 5 and D != 128:
        pytest.skip("FP8 modes: D = 128")
    p = pasa()
    q, k, v = make(B, Hq, Hkv, Sq, Sk, D, kind, 700 + case, **params)
    o_ref, lse_ref = device_result(q, k, v, causal, mode)
    qh, kh, vh = host_tensors(q, k, v)
    units = B * Hkv
    for chunks in sorted({0, 1, 2, 3, units, units + 3}):
        o, lse = p.attn_fwd_host(qh, kh, vh, causal=causal, mode=mode, chunks=chunks)
        p.check_device_error()
        assert torch.equal(o, o_ref), (mode, chunks)
        assert torch.equal(lse, lse_ref), (mode, chunks)


ROW_CASES = [
    # shapes whose automatic plan cuts the first and last unit into query-row pieces
    # (B, Hq, Hkv, Sq, Sk, D, causal, kind, params)
    (1, 64, 1, 2048, 2048, 128, True, "kbias", {"bias_std": 20.0}),       # 6 row pieces
    (1, 64, 1, 2048, 2048 + 256, 64, True, "iid", {}),                    # Sk > Sq by whole blocks
    (1, 64, 1, 2048, 2000, 64, False, "kbias", {"bias_std": 10.0}),       # ragged Sk, no mask
    (2, 32, 2, 2048, 2048, 128, True, "kbias_t3", {"bias_std": 10.0, "t_dof": 3, "t_scale": 4.0}),
]


@pytest.mark.parametrize("case", range(len(ROW_CASES)))
@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4, 5, 6])
def test_host_row_pieces_match_device(case, mode):
    B, Hq, Hkv, Sq, Sk, D, causal, kind, params = ROW_CASES[case]
    if mode >= 5 and D != 128:
        pytest.skip("FP8 modes: D = 128")
    p = pasa()
    plan = p.host_plan(B, Hq, Hkv, Sq, Sk, D, causal, mode, 0)
    assert any(r1 - r0 < Sq for (_, _, r0, r1, _, _) in plan), "the plan has row pieces"
    q, k, v = make(B, Hq, Hkv, Sq, Sk, D, kind, 760 + case, **params)
    o_ref, lse_ref = device_result(q, k, v, causal, mode)
    qh, kh, vh = host_tensors(q, k, v)
    o, lse = p.attn_fwd_host(qh, kh, vh, causal=causal, mode=mode, chunks=0)
    p.check_device_error()
    assert torch.equal(o, o_ref), plan
    assert torch.equal(lse, lse_ref), plan


def test_host_pageable_and_own_buffer():
    p = pasa()
    B, Hq, Hkv, Sq, Sk, D = 2, 8, 4, 520, 520, 128
    q, k, v = make(B, Hq, Hkv, Sq, Sk, D, "kbias", 731, bias_std=20.0)
    o_ref, lse_ref = device_result(q, k, v, True, 0)
    qh, kh, vh = host_tensors(q, k, v, pinned=False)
    out = torch.empty(q.shape, dtype=torch.float16)
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32)
    nbytes = p.host_device_bytes(B, Hq, Hkv, Sq, Sk, D, True, 0, 3)
    buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    p.attn_fwd_host(qh, kh, vh, causal=True, mode=0, out=out, lse=lse, chunks=3, device_buffer=buf)
    assert torch.equal(out, o_ref) and torch.equal(lse, lse_ref)
    # a buffer one byte short is refused before anything is enqueued
    with pytest.raises(p.PasaError):
        p.attn_fwd_host(qh, kh, vh, causal=True, mode=0, out=out, lse=lse, chunks=3, device_buffer=buf[:-1])


def test_host_without_lse():
    p = pasa()
    lib = p.library()
    B, Hq, Hkv, Sq, Sk, D = 1, 4, 2, 300, 300, 64
    q, k, v = make(B, Hq, Hkv, Sq, Sk, D, "iid", 732)
    o_ref, _ = device_result(q, k, v, False, 1)
    qh, kh, vh = host_tensors(q, k, v)
    out = torch.empty(q.shape, dtype=torch.float16).pin_memory()
    P = ctypes.c_void_p
    rc = lib.pasa_attn_fwd_host(P(qh.data_ptr()), P(kh.data_ptr()), P(vh.data_ptr()), P(out.data_ptr()), None, B, Hq,
                                Hkv, Sq, Sk, D, 0, 0.0, 1, 2, None, 0,
                                P(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.current_stream().synchronize()
    assert torch.equal(out, o_ref)


def test_host_calls_queue_in_order_on_one_buffer():
    """Back-to-back calls without a host synchronisation, sharing one device buffer: each
    call's copies wait for the work queued before it, so neither result is overwritten."""
    p = pasa()
    B, Hq, Hkv, Sq, Sk, D = 2, 8, 4, 1030, 1030, 128
    ins = [make(B, Hq, Hkv, Sq, Sk, D, "kbias", 740 + i, bias_std=10.0) for i in range(3)]
    refs = [device_result(*x, True, 0) for x in ins]
    buf = torch.empty(p.host_device_bytes(B, Hq, Hkv, Sq, Sk, D, True, 0, 4), dtype=torch.uint8, device="cuda")
    outs = []
    for x in ins:
        qh, kh, vh = host_tensors(*x)
        outs.append(p.attn_fwd_host(qh, kh, vh, causal=True, mode=0, chunks=4, device_buffer=buf, sync=False))
    torch.cuda.current_stream().synchronize()
    p.check_device_error()
    for (o, lse), (o_ref, lse_ref) in zip(outs, refs):
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    # the same with row pieces sharing a unit's key slot
    B, Hq, Hkv, Sq, Sk, D = 1, 64, 1, 2048, 2048, 128
    ins = [make(B, Hq, Hkv, Sq, Sk, D, "kbias", 750 + i, bias_std=10.0) for i in range(2)]
    refs = [device_result(*x, True, 1) for x in ins]
    buf = torch.empty(p.host_device_bytes(B, Hq, Hkv, Sq, Sk, D, True, 1, 0), dtype=torch.uint8, device="cuda")
    outs = []
    for x in ins:
        qh, kh, vh = host_tensors(*x)
        outs.append(p.attn_fwd_host(qh, kh, vh, causal=True, mode=1, device_buffer=buf, sync=False))
    torch.cuda.current_stream().synchronize()
    for (o, lse), (o_ref, lse_ref) in zip(outs, refs):
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


def test_release_host_streams_then_call_again():
    """pasa_release_host_streams drops the side streams (after their work is done); the
    next host call creates them again and still agrees bit for bit. Releasing twice, or
    before any host call, is a no-op."""
    p = pasa()
    B, Hq, Hkv, Sq, Sk, D = 2, 6, 3, 400, 400, 128
    q, k, v = make(B, Hq, Hkv, Sq, Sk, D, "kbias", 734, bias_std=20.0)
    o_ref, lse_ref = device_result(q, k, v, True, 0)
    qh, kh, vh = host_tensors(q, k, v)
    o1, l1 = p.attn_fwd_host(qh, kh, vh, causal=True, mode=0, chunks=3, sync=False)
    p.release_host_streams()   # waits for the side streams' share of the call above
    torch.cuda.current_stream().synchronize()
    assert torch.equal(o1, o_ref) and torch.equal(l1, lse_ref)
    p.release_host_streams()
    o2, l2 = p.attn_fwd_host(qh, kh, vh, causal=True, mode=0, chunks=3)
    assert torch.equal(o2, o_ref) and torch.equal(l2, lse_ref)
    p.release_host_streams()
    p.check_device_error()


def test_host_against_oracle():
    p = pasa()
    B, Hq, Hkv, Sq, Sk, D = 2, 4, 2, 333, 333, 128
    q, k, v = make(B, Hq, Hkv, Sq, Sk, D, "kbias", 733, bias_std=20.0)
    qh, kh, vh = host_tensors(q, k, v)
    o, lse = p.attn_fwd_host(qh, kh, vh, causal=True, mode=0, chunks=0)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=True)
    rmse, _ = rel_errors(o.double().numpy(), o_ref)
    assert rmse <= 5e-3
    assert np.all(np.isfinite(o.float().numpy()))
    tol = lse_tolerance(q, k, True, 0, D)
    assert np.max(np.abs(lse.double().numpy() - lse_ref)) <= tol


def test_host_full_size_32k_matches_device():
    """The call the end-to-end benchmark times, at full size (32K biased causal workload,
    B1 Hq28/Hkv4 D128, mode 0, automatic plan with row pieces): bit-identical to the
    device-resident call."""
    p = pasa()
    w = wl.WORKLOADS["kbias10_t3_b1h28g4_s32768_d128_causal"]
    q, k, v = wl.make_inputs(w)
    plan = p.host_plan(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, w.causal, 0, 0)
    assert len(plan) == 10
    o_ref, lse_ref = device_result(q, k, v, w.causal, 0)
    qh, kh, vh = host_tensors(q, k, v)
    o, lse = p.attn_fwd_host(qh, kh, vh, causal=w.causal, mode=0)
    p.check_device_error()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    assert bool(torch.isfinite(o).all())
