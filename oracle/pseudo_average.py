"""Reference for the per-key-block pseudo-average and the shifted keys (numpy, exact).

TEST INFRASTRUCTURE ONLY: the product path never imports this module.

Source: "Online Pseudo-average Shifting Attention (PASA) for Robust Low-precision LLM
Inference" (arXiv 2503.01873), Abstract. The abstract names "online pseudo-average
shifting" and says the algorithm stays mathematically equivalent to plain attention; it
does not define the pseudo-average. Because the offsets q_i . m_j are added back
("global recovering"), any per-channel vector m_j keeps the result exact, so the choice
only affects rounding. The reading implemented here (the CUDA kernel implements the
same reading independently):

For key block j (rows j*Bn .. min(Sk, (j+1)*Bn) - 1, n valid rows) and channel d:

1. M   = max_r |K[r, d]|, an fp16 value.
2. g   = the spacing of fp16 numbers at M (its unit in the last place): 2^(E-25) for
         biased exponent E >= 1, and 2^-24 for subnormal M or M = 0.
3. t_r = round-half-even(K[r, d] / g), an integer with |t_r| <= 2047.
4. m   = g * round-half-even(sum_r t_r / n), computed in exact integer arithmetic.
   The result lies on the grid g, so |m| <= M and m is exactly an fp16 value.
5. If E >= 30 (M >= 32768) or K holds inf/NaN in that block and channel, m = 0, so that
   the shifted value K - m can never leave the fp16 range.
6. K'[r, d] = fp16(K[r, d] - m), rounded to nearest even once.

It is a "pseudo" average: the mean of K rounded to the grid of the block's largest
magnitude. Because m sits on that grid, K - m is exact in fp16 for most elements, so
shifting loses almost nothing even when the true mean is near zero. Parity for this
function is pinned by closed forms and bounds in tests/test_pseudo_average_oracle.py.

The alternative reading kept beside it (``rule="plain"``): steps 2-4 replaced by
m = fp16(exact mean of the block's n values), rounded to nearest even once; the guard of
step 5 and step 6 are the same. That is the plain fp16-rounded block mean, which the
grid reading is compared against.
"""
from __future__ import annotations

import numpy as np


def block_rows_for(D: int) -> int:
    """Keys per block for head dim D: 128.

    The Abstract leaves the block length open; the reading here is that the shift block is
    the attention kernel's key tile, so its length is whatever that tile is for the head dim.
    """
    return 128


def grid_step(absmax: np.ndarray) -> np.ndarray:
    """fp16 unit in the last place at each (non-negative) fp16 value, as float64 (step 2)."""
    bits = np.asarray(absmax, dtype=np.float16).view(np.uint16).astype(np.int64) & 0x7FFF
    e = bits >> 10
    return np.where(e >= 1, np.ldexp(1.0, (e - 25).astype(np.int64)), np.ldexp(1.0, -24))


def _round_half_even_div(num: np.ndarray, den: np.ndarray) -> np.ndarray:
    """round-half-even(num / den) for integer arrays, den > 0, in exact integer arithmetic."""
    a = np.abs(num)
    q = a // den
    r = a - q * den
    up = (2 * r > den) | ((2 * r == den) & (q % 2 == 1))
    q = q + up.astype(np.int64)
    return np.where(num < 0, -q, q)


def fp16_round_rational(num: int, den: int) -> float:
    """num / den (Python integers, den > 0) rounded to the nearest fp16 value, ties to even,
    in exact integer arithmetic. The magnitude must stay below 65520 (no overflow)."""
    if num == 0:
        return 0.0
    a = abs(num)
    k = a.bit_length() - den.bit_length()          # 2^k <= a / den < 2^(k+1) after the fix-up
    if (a << max(0, -k)) < (den << max(0, k)):
        k -= 1
    u = max(k - 10, -24)                           # exponent of the fp16 spacing at a / den
    n2, d2 = (a, den << u) if u >= 0 else (a << -u, den)
    q, r = divmod(n2, d2)
    if 2 * r > d2 or (2 * r == d2 and q % 2 == 1):
        q += 1
    return float(np.ldexp(float(q), u)) * (1.0 if num > 0 else -1.0)


def block_pseudo_average(kb: np.ndarray, rule: str = "grid") -> np.ndarray:
    """Pseudo-average of one key block ``kb`` [n, D] fp16 (steps 1-5; ``rule="plain"``: the
    exact block mean rounded once to fp16). Returns [D] fp16."""
    kb = np.asarray(kb, dtype=np.float16)
    n = kb.shape[0]
    if n == 0:
        return np.zeros(kb.shape[1], np.float16)
    x = kb.astype(np.float64)
    finite = np.all(np.isfinite(x), axis=0)
    xm = np.where(np.isfinite(x), x, 0.0)
    M = np.max(np.abs(xm), axis=0).astype(np.float16)
    bits = M.view(np.uint16).astype(np.int64) & 0x7FFF
    E = bits >> 10
    if rule == "plain":
        # every fp16 value is an integer multiple of 2^-24: the sum is an exact integer
        units = [int(v) for v in np.sum(np.rint(np.ldexp(xm, 24)).astype(np.int64), axis=0)]
        m = np.array([fp16_round_rational(s_, n << 24) for s_ in units])
    elif rule == "grid":
        g = grid_step(M)
        t = np.rint(xm / g).astype(np.int64)            # exact: g is a power of two
        s = np.sum(t, axis=0)
        mu = _round_half_even_div(s, np.full_like(s, n))
        m = mu.astype(np.float64) * g
    else:
        raise ValueError(rule)
    m = np.where((E >= 30) | ~finite, 0.0, m)
    out = m.astype(np.float16)
    assert np.all(out.astype(np.float64) == m), "pseudo-average must be an exact fp16 value"
    return out


def kshift(k: np.ndarray, block_rows: int | None = None, rule: str = "grid"):
    """Shift every key block by its pseudo-average (``rule`` as in block_pseudo_average).

    k: [B, H, Sk, D] fp16. Returns (k_shifted [B, H, Sk, D] fp16,
    means [B, H, ceil(Sk / block_rows), D] fp16).
    """
    k = np.asarray(k, dtype=np.float16)
    B, H, Sk, D = k.shape
    block_rows = block_rows_for(D) if block_rows is None else block_rows
    nb = (Sk + block_rows - 1) // block_rows
    means = np.zeros((B, H, nb, D), np.float16)
    ks = np.empty_like(k)
    for b in range(B):
        for h in range(H):
            for j in range(nb):
                r0, r1 = j * block_rows, min(Sk, (j + 1) * block_rows)
                m = block_pseudo_average(k[b, h, r0:r1], rule)
                means[b, h, j] = m
                ks[b, h, r0:r1] = (k[b, h, r0:r1].astype(np.float64) - m.astype(np.float64)).astype(np.float16)
    return ks, means


def kshift_fast(k: np.ndarray, block_rows: int | None = None, rule: str = "grid"):
    """Same result as :func:`kshift`, vectorised over all blocks (for large inputs).

    rule="plain" rounds the exact mean S / n (S the exact sum, an integer multiple of
    2^-24 below 2^22) through float64 and then to fp16. That equals one rounding of the
    exact mean: a value S / (n 2^24) that is not itself an fp16 tie lies at least
    2^-25 / n >= 2^-32 from every tie (ties are multiples of 2^-25), while the float64
    division errs by at most 2^-53 * 2^15 = 2^-38."""
    k = np.asarray(k, dtype=np.float16)
    B, H, Sk, D = k.shape
    block_rows = block_rows_for(D) if block_rows is None else block_rows
    nb = (Sk + block_rows - 1) // block_rows
    pad = nb * block_rows - Sk
    x = k.astype(np.float64)
    valid = np.ones((nb * block_rows,), bool)
    if pad:
        x = np.concatenate([x, np.zeros((B, H, pad, D))], axis=2)
        valid[Sk:] = False
    x = x.reshape(B, H, nb, block_rows, D)
    vmask = valid.reshape(nb, block_rows)[None, None, :, :, None]
    fin = np.isfinite(x)
    finite = np.all(fin | ~vmask, axis=3)
    xm = np.where(fin & vmask, x, 0.0)
    M = np.max(np.abs(xm), axis=3).astype(np.float16)
    E = (M.view(np.uint16).astype(np.int64) & 0x7FFF) >> 10
    n = np.minimum(block_rows, Sk - np.arange(nb) * block_rows).astype(np.int64)
    if rule == "plain":
        s = np.sum(np.rint(np.ldexp(xm, 24)).astype(np.int64), axis=3)
        mean = s.astype(np.float64) / n[None, None, :, None]
        mplain = np.ldexp(mean, -24).astype(np.float16).astype(np.float64)
        m = np.where((E >= 30) | ~finite, 0.0, mplain)
    elif rule == "grid":
        g = grid_step(M)
        t = np.rint(xm / g[:, :, :, None, :]).astype(np.int64)
        s = np.sum(t, axis=3)
        mu = _round_half_even_div(s, np.broadcast_to(n[None, None, :, None], s.shape))
        m = np.where((E >= 30) | ~finite, 0.0, mu.astype(np.float64) * g)
    else:
        raise ValueError(rule)
    means = m.astype(np.float16)
    ks = (x - means.astype(np.float64)[:, :, :, None, :]).reshape(B, H, nb * block_rows, D)[:, :, :Sk]
    return ks.astype(np.float16), means
