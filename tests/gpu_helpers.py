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


def _f16_spacing(x):
    """Spacing of fp16 numbers at |x| (2^(e-10) for normal magnitudes, 2^-24 below 2^-14)."""
    a = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -24)))
    return np.where(a >= 2.0 ** -14, np.ldexp(1.0, (e - 10).astype(np.int64)), 2.0 ** -24)


def f16_score_rmse_model(q, k, v, causal, mode, rows):
    """Predicted relRMSE of O from fp16 accumulation of the scores (modes 0, 2 and 4).

    Model. The score MMA accumulates S'_ij = q_i . k'_j in fp16 (k' = K' in the shifted
    modes, K in the naive one) over D / 16 instructions of 16 channels, each ending in one
    round-to-nearest of the accumulator. A rounding at magnitude |s| errs by a value spread
    evenly over +-u/2, u = fp16 spacing at |s|, i.e. with variance u^2 / 12. Taking the
    spacing at the final |S'_ij| for every step (where the scores are large, which is where
    the error matters, the partial sums grow to that size), each score's error has variance
    sigma_ij^2 = scale^2 * (D / 16) * u(S'_ij)^2 / 12, independently across keys. To first
    order O_i moves by sum_j p_ij delta_ij (v_j - O_i), so the expected square
    error of element (i, d) is sum_j p_ij^2 sigma_ij^2 (v_jd - O_id)^2. The prediction is the
    square root of its mean over the sampled rows and channels, over RMS(O_ref).

    Mode 4 adds its fp16 PV accumulator: 8 roundings per 128-key block of values of about
    the size of l * O plus about 20 for the row sum, each of relative variance 2^-22 / 12,
    i.e. 2^-11 * sqrt((8 * nblk + 20) / 12) relative to RMS(O).

    rows: flat (b * Hq + h) * Sq + i indices. Returns the predicted relRMSE."""
    from oracle import pseudo_average as pa

    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = k.shape
    g = Hq // Hkv
    scale = 1.0 / math.sqrt(D)
    bn = pa.block_rows_for(D)
    if mode in (0, 4):
        kk, means = pa.kshift_fast(k)
    elif mode == 2:
        kk, means = k, None
    else:
        raise ValueError("the model covers the fp16-accumulated score modes 0, 2 and 4")
    num = den = 0.0
    for r in np.asarray(rows, np.int64):
        b, rem = divmod(int(r), Hq * Sq)
        h, i = divmod(rem, Sq)
        hk = h // g
        lim = min(Sk, i + Sk - Sq + 1) if causal else Sk
        if lim <= 0:
            continue
        qi = q[b, h, i].astype(np.float64)
        sp = kk[b, hk, :lim].astype(np.float64) @ qi
        s = sp if means is None else sp + np.repeat(means[b, hk].astype(np.float64), bn, axis=0)[:lim] @ qi
        s = scale * s
        p = np.exp(s - s.max())
        p /= p.sum()
        vv = v[b, hk, :lim].astype(np.float64)
        o = p @ vv
        sig2 = scale ** 2 * (D // 16) * _f16_spacing(sp) ** 2 / 12.0
        num += float(((p * p * sig2)[:, None] * (vv - o) ** 2).sum())
        den += float((o * o).sum())
    pred = math.sqrt(num / max(den, 1e-300))
    if mode == 4:
        pred += 2.0 ** -11 * math.sqrt((8 * (-(-Sk // 128)) + 20) / 12.0)
    return pred


# Gate on the model: the measured relRMSE may not exceed 2 x the prediction plus the
# fp32-score modes' own error level (P rounded to fp16, ex2.approx, fp32 sums). On the
# measured workloads the GPU's fp16-score error is 0.5-0.95 x the prediction, and an
# emulated round-to-nearest accumulator on small samples 0.3-1.3 x.
F16_MODEL_FACTOR = 2.0
F16_MODEL_FLOOR = 5e-4


def f16_score_rmse_gate(pred):
    return F16_MODEL_FACTOR * pred + F16_MODEL_FLOOR
