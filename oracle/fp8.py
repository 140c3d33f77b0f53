"""FP8 (e4m3) reference for the FP8 score modes. TEST INFRASTRUCTURE ONLY.

"Online Pseudo-average Shifting Attention (PASA) for Robust Low-precision LLM Inference"
(arXiv 2503.01873), Abstract: the shift keeps low-precision attention scores in range. The
FP8 modes carry that to 8-bit scores: Q and the (shifted) keys are quantised to e4m3, the
score GEMM accumulates in fp32, and everything after it is the fp32-score PASA path.

e4m3 (the "fn" variant): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; no
infinities; largest finite value 1.75 * 2^8 = 448; smallest normal 2^-6; subnormals
k * 2^-9 for k = 1..7. Rounding is to nearest, ties to even, and values beyond 448
saturate to 448 (the kernel's cvt.rn.satfinite).

Scales. A row of Q (per query row) or a 128-key block of keys (all channels) with absolute
maximum a is stored as codes t = e4m3(x * inv) with inv = fp32(448 / a), and read back as
t * s with s = fp32(a / 448); a = 0 gives inv = s = 1. Both divisions and the product
x * inv are single fp32 roundings, as in the kernel, so the codes here and on the GPU are
the same numbers.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_round(x) -> np.ndarray:
    """Nearest e4m3 value (ties to even, saturating at +-448), as float64."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    # exponent of the binade, clamped below at the normal range (subnormals share 2^-9 spacing)
    _, e = np.frexp(np.where(a > 0, a, 1.0))        # a = f * 2^e, f in [0.5, 1)
    e = np.maximum(e - 1, -6)                        # a in [2^e, 2^(e+1))
    step = np.ldexp(1.0, e - 3)                      # 3 mantissa bits
    q = np.rint(a / step) * step                     # exact: a / step is a small integer + fraction
    q = np.minimum(q, E4M3_MAX)
    return np.copysign(q, x)


def scales(absmax):
    """(inv, s) in fp32 for absolute maxima `absmax` (see the module docstring)."""
    a = np.asarray(absmax, dtype=np.float32)
    safe = np.where(a > 0, a, np.float32(1.0)).astype(np.float32)
    inv = np.where(a > 0, np.float32(E4M3_MAX) / safe, np.float32(1.0)).astype(np.float32)
    s = np.where(a > 0, safe / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    return inv, s


def quantize_rows(q):
    """Q [B, H, S, D] fp16 -> (codes as float64 e4m3 values, per-row scale s [B, H, S] fp32)."""
    x = np.asarray(q, dtype=np.float16).astype(np.float32)
    inv, s = scales(np.abs(x).max(axis=-1))
    t = (x * inv[..., None]).astype(np.float32)      # one fp32 rounding
    return e4m3_round(t), s


def quantize_blocks(k, block_rows: int = 128):
    """K [B, H, S, D] fp16 -> (codes as float64, per-block scale s [B, H, ceil(S / block_rows)] fp32)."""
    x = np.asarray(k, dtype=np.float16).astype(np.float32)
    B, H, S, D = x.shape
    nb = -(-S // block_rows)
    pad = np.zeros((B, H, nb * block_rows - S, D), np.float32)
    xb = np.concatenate([x, pad], axis=2).reshape(B, H, nb, block_rows, D)
    inv, s = scales(np.abs(xb).max(axis=(3, 4)))
    t = (xb * inv[..., None, None]).astype(np.float32)
    codes = e4m3_round(t).reshape(B, H, nb * block_rows, D)[:, :, :S]
    return codes, s


def attention_fp8(q, k, v, causal: bool, means=None, block_rows: int = 128, scale=None):
    """fp64 attention on the dequantised e4m3 Q and keys, plus the offsets q . m_j (fp16 q and
    means, exact in fp64) when means is given: the number the FP8 modes compute, up to fp32
    accumulation and the fp16 rounding of P. q [B,Hq,Sq,D], k (shifted or raw) and v
    [B,Hkv,Sk,D] fp16. Dense numpy; for small sizes only. Returns (o, lse) in float64."""
    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = k.shape
    g = Hq // Hkv
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    q8, sq = quantize_rows(q)
    k8, sk = quantize_blocks(k, block_rows)
    qd = q8 * sq.astype(np.float64)[..., None]
    kd = k8 * np.repeat(sk.astype(np.float64), block_rows, axis=2)[:, :, :Sk, None]
    kd = np.repeat(kd, g, axis=1)
    s = qd @ kd.transpose(0, 1, 3, 2)
    if means is not None:
        mrow = np.repeat(np.repeat(means.astype(np.float64), block_rows, axis=2)[:, :, :Sk], g, axis=1)
        s = s + q.astype(np.float64) @ mrow.transpose(0, 1, 3, 2)
    s = s * scale
    if causal:
        mask = np.arange(Sk)[None, :] <= np.arange(Sq)[:, None] + (Sk - Sq)
        s = np.where(mask, s, -np.inf)
    mx = s.max(axis=-1, keepdims=True)
    fin = np.isfinite(mx)
    p = np.where(fin, np.exp(s - np.where(fin, mx, 0.0)), 0.0)
    l = p.sum(axis=-1, keepdims=True)
    vv = np.repeat(v.astype(np.float64), g, axis=1)
    o = np.where(l > 0, (p @ vv) / np.where(l > 0, l, 1.0), 0.0)
    lse = np.where(l[..., 0] > 0, mx[..., 0] + np.log(np.where(l[..., 0] > 0, l[..., 0], 1.0)), -np.inf)
    return o, lse
