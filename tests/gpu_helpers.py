"""Shared helpers for the GPU tests: device upload and error metrics.

Error metrics (output scale): relRMSE = RMS(O - O_ref) / RMS(O_ref) and
relMax = max |O - O_ref| / max |O_ref| over the compared elements.
"""
import math

import numpy as np
import torch

import oracle


def to_dev(*xs):
    return [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in xs]


def rel_errors(o_gpu, o_ref):
    o_gpu = np.asarray(o_gpu, np.float64)
    o_ref = np.asarray(o_ref, np.float64)
    d = o_gpu - o_ref
    rmse = float(np.sqrt(np.mean(d * d)) / max(np.sqrt(np.mean(o_ref * o_ref)), 1e-300))
    rmax = float(np.max(np.abs(d)) / max(np.max(np.abs(o_ref)), 1e-300))
    return rmse, rmax


def gather_rows(o, rows):
    """Rows (flat (b*H + h)*S + i indices) of a [B,H,S,D] device tensor, as float64 numpy."""
    D = o.shape[-1]
    flat = o.reshape(-1, D)
    idx = torch.as_tensor(rows, device=o.device, dtype=torch.long)
    return flat.index_select(0, idx).double().cpu().numpy()


def lse_tolerance(q, k, causal, mode, D):
    """LSE bound derived from the arithmetic. LSE is 1-Lipschitz in the max norm of the
    scores, so it moves by at most scale * max_ij |delta S_ij|:
      * shifted modes: K' = fp16(K - m) is not always exact; the oracle knows its rounding
        error E = K' - (K - m) exactly, and the score moves by q_i . E_j;
      * fp16-accumulated modes: a few units of the fp16 spacing at the largest score
        magnitude (of the shifted keys for mode 0, of the raw keys for mode 2);
      * plus 2e-3 for fp32 accumulation, ex2.approx and fp16 rounding of P."""
    from oracle import pseudo_average as pa

    scale = 1.0 / math.sqrt(D)
    g = q.shape[1] // k.shape[1]
    qd = q.astype(np.float64)
    tol = 2e-3
    ks = None
    if mode in (0, 1, 4):
        ks, means = pa.kshift_fast(k)
        rows = np.repeat(means.astype(np.float64), pa.block_rows_for(k.shape[3]), axis=2)[:, :, :k.shape[2]]
        err = ks.astype(np.float64) - (k.astype(np.float64) - rows)
        err = np.repeat(err, g, axis=1)
        tol += scale * float(np.abs(qd @ err.transpose(0, 1, 3, 2)).max())
    if mode in (0, 2, 4):
        kk = ks if mode in (0, 4) else k
        smax = float(oracle.row_max_abs_score(q, kk, causal).max())
        ulp = 2.0 ** (math.floor(math.log2(max(smax, 1e-30))) - 10)
        tol += 4.0 * ulp * scale
    if mode == 4:
        tol += f16all_bound(k.shape[2])   # fp16 running row sum: ln(1 + x) <= x
    return tol


def f16all_bound(Sk):
    """Mode 4 (fp16 PV accumulator and fp16 running row sum), relative to max |v| for O and
    to 1 for the LSE. Each of the 8 PV MMA steps of a 128-key block rounds the accumulator
    to fp16 once (at most 2^-11 of a value bounded by l * max|v|); each block's row sum
    takes about 20 fp16 additions and one more to join l. Over nblk blocks that is at most
    (9 * nblk + 20) roundings of relative size 2^-11."""
    nblk = -(-Sk // 128)
    return (9 * nblk + 20) * 2.0 ** -11
