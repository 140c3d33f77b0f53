"""GPU: pasa_attn_fwd_noalloc, the entry point for callers that cannot allocate device memory.

Such callers (a process whose GPU memory a framework or serving allocator has reserved up
front, or a latency-bound loop where allocation is not allowed) get the shifted keys and
block means placed in a fixed 64 MiB array inside the library instead of a workspace.
This checks, through the C ABI, that two calls in a row give the same output as the
workspace entry point within the parity tolerances, and that oversized problems are
refused before anything is launched. The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu

PASA_ERR_WORKSPACE = -7


def _lib():
    import precision_flashattention_numerics_gb300 as pasa

    return pasa, pasa.library()


def _noalloc(lib, q, k, v, causal, mode):
    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = k.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Sq), device=q.device, dtype=torch.float32)
    P = ctypes.c_void_p
    rc = lib.pasa_attn_fwd_noalloc(P(q.data_ptr()), P(k.data_ptr()), P(v.data_ptr()), P(o.data_ptr()),
                                   P(lse.data_ptr()), B, Hq, Hkv, Sq, Sk, D, int(causal), 0.0, mode,
                                   P(torch.cuda.current_stream().cuda_stream))
    return rc, o, lse


def _rel(a, b):
    a = a.double()
    b = b.double()
    d = a - b
    return (d.square().mean().sqrt() / b.square().mean().sqrt()).item(), (d.abs().max() / b.abs().max()).item()


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    pasa, lib = _lib()
    cases = [
        (wl.Workload("na0", 1, 8, 2, 700, 700, 128, True, "kbias", 901, (("bias_std", 20.0),)), 0),
        (wl.Workload("na1", 2, 3, 3, 450, 333, 64, False, "iid", 902), 1),
    ]
    for w, mode in cases:
        q, k, v = (torch.from_numpy(x).cuda() for x in wl.make_inputs(w))
        o_ref, lse_ref = pasa.attn_fwd(q, k, v, causal=w.causal, mode=mode)
        rc, o, lse = _noalloc(lib, q, k, v, w.causal, mode)
        assert rc == 0, lib.pasa_strerror(rc)
        pasa.check_device_error()
        assert torch.isfinite(o).all()
        rmse, rmax = _rel(o, o_ref)
        assert rmse <= 2e-3 and rmax <= 1e-2, (rmse, rmax)
        assert (lse - lse_ref).abs().max().item() <= 2e-3


def test_noalloc_refuses_problems_larger_than_its_scratch():
    pasa, lib = _lib()
    # keys of 1 x 1 x 262200 x 128 fp16 need just over 64 MiB of shifted keys: refused on the host
    Sk, D = 262200, 128
    assert lib.pasa_attn_fwd_workspace_bytes(1, 1, Sk, D, 0) > (64 << 20)
    q = torch.zeros((1, 1, 128, D), device="cuda", dtype=torch.float16)
    k = torch.zeros((1, 1, Sk, D), device="cuda", dtype=torch.float16)
    v = torch.zeros_like(k)
    rc, _, _ = _noalloc(lib, q, k, v, False, 0)
    assert rc == PASA_ERR_WORKSPACE
    # the modes without the shift need no scratch and run at any size
    rc, o, _ = _noalloc(lib, q, k, v, False, 3)
    assert rc == 0
    pasa.check_device_error()
    assert torch.count_nonzero(o).item() == 0
