"""Failure detection on the GPU, without a fault.

Every wait in the library's kernels is bounded: after a limit it records a timeout in a
device error word and the kernel returns, so the host can read the error and the context
stays usable. pasa_selftest_wait_timeout runs that wait on a barrier nothing arrives on;
this test checks the status the host reads, the site tag, that the word is cleared, and
that the next attention call is correct (checked against the fp64 oracle). A timeout ends
only the CTA it happened in: a later launch is correct even while the timeout is still unread.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_helpers import rel_errors, to_dev

pytestmark = pytest.mark.gpu

SELFTEST_SITE = 0x5E1F7E57
PASA_ERR_TIMEOUT = -6


def test_bounded_wait_gives_up_reports_and_clears():
    import precision_flashattention_numerics_gb300 as p

    lib = p.library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    info = ctypes.c_ulonglong(0)
    assert lib.pasa_check_device_error(stream, ctypes.byref(info)) == 0, "an error was already pending"

    t0 = time.monotonic()
    p.selftest_wait_timeout()
    rc = lib.pasa_check_device_error(stream, ctypes.byref(info))
    elapsed = time.monotonic() - t0
    assert rc == PASA_ERR_TIMEOUT
    assert info.value & 0xFFFFFFFF == SELFTEST_SITE
    assert 1.5 < elapsed < 60.0, elapsed        # gave up at its 2 s limit: not at once, not never
    # read once, the word is clear again
    assert lib.pasa_check_device_error(stream, ctypes.byref(info)) == 0

    # the context is usable: the full path still computes attention correctly
    w = wl.Workload("after_timeout", 1, 4, 2, 300, 300, 128, True, "kbias", 790, (("bias_std", 20.0),))
    q, k, v = wl.make_inputs(w)
    qt, kt, vt = to_dev(q, k, v)
    o, lse = p.attn_fwd(qt, kt, vt, causal=True, mode=1)
    p.check_device_error()
    o_ref, _ = oracle.attention(q, k, v, causal=True)
    rmse, rmax = rel_errors(o.double().cpu().numpy(), o_ref)
    assert rmse <= 5e-3 and np.isfinite(o.float().cpu().numpy()).all()


def test_python_check_raises_the_timeout():
    import precision_flashattention_numerics_gb300 as p

    p.check_device_error()
    p.selftest_wait_timeout()
    with pytest.raises(p.PasaError) as exc:
        p.check_device_error()
    assert exc.value.status == PASA_ERR_TIMEOUT
    p.check_device_error()   # cleared


def test_unread_timeout_does_not_abort_later_launches():
    # The error word latches the timeout until it is read, but no kernel reads it: a wait
    # gives up only at its own limit or when another warp of its CTA has given up. The
    # attention call queued behind an unread timeout must still be correct, and the timeout
    # must still be reported.
    import precision_flashattention_numerics_gb300 as p

    lib = p.library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    info = ctypes.c_ulonglong(0)
    assert lib.pasa_check_device_error(stream, ctypes.byref(info)) == 0, "an error was already pending"
    p.selftest_wait_timeout()
    w = wl.Workload("behind_timeout", 1, 8, 2, 1000, 1000, 128, True, "kbias", 791, (("bias_std", 20.0),))
    q, k, v = wl.make_inputs(w)
    qt, kt, vt = to_dev(q, k, v)
    o, lse = p.attn_fwd(qt, kt, vt, causal=True, mode=0)      # queued behind the timed-out kernel
    torch.cuda.synchronize()
    rc = lib.pasa_check_device_error(stream, ctypes.byref(info))
    assert rc == PASA_ERR_TIMEOUT and info.value & 0xFFFFFFFF == SELFTEST_SITE
    o_ref, lse_ref = oracle.attention(q, k, v, causal=True)
    rmse, rmax = rel_errors(o.double().cpu().numpy(), o_ref)
    assert rmse <= 5e-3 and rmax <= 5e-2, (rmse, rmax)
    assert np.abs(lse.double().cpu().numpy() - lse_ref).max() <= 1e-2
    assert lib.pasa_check_device_error(stream, ctypes.byref(info)) == 0
