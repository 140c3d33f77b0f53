/*
 * Plain fp64 CPU attention: the reference every GPU result is compared with.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may load or call this file:
 * only the tests, the package's smoke check and the bench's CPU-baseline leg do.
 * It shares no code, header or constant with the CUDA library.
 *
 * What it computes. "Online Pseudo-average Shifting Attention (PASA) for Robust
 * Low-precision LLM Inference" (arXiv 2503.01873), Abstract: PASA is a low-precision
 * algorithm, based on Flash Attention, that is mathematically equivalent to plain
 * attention. So the reference is the plain definition, with no blocking and no
 * shifting, on the exact values of the fp16 inputs:
 *
 *     s_ij  = scale * sum_d q_id k_jd            (j visible: all j, or j <= i + Sk - Sq when causal)
 *     O_i   = sum_j exp(s_ij - max_j s_ij) v_j / sum_j exp(s_ij - max_j s_ij)
 *     LSE_i = max_j s_ij + ln sum_j exp(s_ij - max_j s_ij)
 *
 * A row with no visible key gets O_i = 0 and LSE_i = -inf.
 *
 * Layout: q [B, Hq, Sq, D], k and v [B, Hkv, Sk, D], as raw IEEE binary16 bit patterns;
 * query head h reads key/value head h / (Hq / Hkv). Rows are addressed by the flat
 * index g = (b*Hq + h)*Sq + i. Outputs are fp64: o [n_rows, D], lse [n_rows].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* binary16 -> double, exact: decoded from sign, exponent and fraction fields. */
static double half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                /* zero or subnormal */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f | 0x400), e - 25);   /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

static double g_h2d[65536];
static int g_h2d_ready = 0;

static void init_table(void) {
    if (g_h2d_ready) return;
    for (int i = 0; i < 65536; ++i) g_h2d[i] = half_to_double((uint16_t)i);
    g_h2d_ready = 1;
}

double oracle_half_to_double(uint16_t h) { return half_to_double(h); }

/* Number of keys visible to query row i. */
static int64_t visible_keys(int64_t i, int64_t Sq, int64_t Sk, int causal) {
    if (!causal) return Sk;
    int64_t n = i + Sk - Sq + 1;
    if (n < 0) n = 0;
    if (n > Sk) n = Sk;
    return n;
}

/*
 * Optional per-block offsets (the "global recovering" reading): when `means` is not
 * NULL, `k` holds shifted keys k'_j and the score of key j adds back q_i . m_{j / bn},
 * where means is [B, Hkv, ceil(Sk/bn), D] fp16 bits. With means == NULL this is the
 * plain definition above.
 */
static void attention_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                           const uint16_t *means, int64_t bn,
                           double *o, double *lse,
                           int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk, int64_t D,
                           int causal, double scale, const int64_t *rows, int64_t n_rows) {
    init_table();
    int64_t group = Hq / Hkv;
    int64_t nb = bn > 0 ? (Sk + bn - 1) / bn : 0;
    (void)B;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
        double *qr = (double *)malloc(sizeof(double) * (size_t)D);
        double *acc = (double *)malloc(sizeof(double) * (size_t)D);
        double *cj = (double *)malloc(sizeof(double) * (size_t)(nb > 0 ? nb : 1));
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < n_rows; ++r) {
            int64_t g = rows ? rows[r] : r;
            int64_t i = g % Sq;
            int64_t h = (g / Sq) % Hq;
            int64_t b = g / (Sq * Hq);
            int64_t hk = h / group;
            const uint16_t *qrow = q + g * D;
            const uint16_t *kh = k + (b * Hkv + hk) * Sk * D;
            const uint16_t *vh = v + (b * Hkv + hk) * Sk * D;
            for (int64_t d = 0; d < D; ++d) qr[d] = g_h2d[qrow[d]];
            int64_t n = visible_keys(i, Sq, Sk, causal);
            double *orow = o + r * D;
            if (n == 0) {
                for (int64_t d = 0; d < D; ++d) orow[d] = 0.0;
                lse[r] = -INFINITY;
                continue;
            }
            if (means) {
                const uint16_t *mh = means + (b * Hkv + hk) * nb * D;
                for (int64_t jb = 0; jb < nb; ++jb) {
                    double c = 0.0;
                    for (int64_t d = 0; d < D; ++d) c += qr[d] * g_h2d[mh[jb * D + d]];
                    cj[jb] = c;
                }
            }
            /* pass 1: scores and their maximum */
            double mx = -INFINITY;
            for (int64_t j = 0; j < n; ++j) {
                const uint16_t *kr = kh + j * D;
                double dot = 0.0;
                for (int64_t d = 0; d < D; ++d) dot += qr[d] * g_h2d[kr[d]];
                if (means) dot += cj[j / bn];
                s[j] = scale * dot;
                if (s[j] > mx) mx = s[j];
            }
            /* pass 2: exponentials, their sum, and the weighted sum of values */
            double l = 0.0;
            for (int64_t d = 0; d < D; ++d) acc[d] = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                double p = exp(s[j] - mx);
                l += p;
                const uint16_t *vr = vh + j * D;
                for (int64_t d = 0; d < D; ++d) acc[d] += p * g_h2d[vr[d]];
            }
            for (int64_t d = 0; d < D; ++d) orow[d] = acc[d] / l;
            lse[r] = mx + log(l);
        }
        free(s);
        free(qr);
        free(acc);
        free(cj);
    }
}

/* Plain attention (the definition in the header comment). rows == NULL: every row. */
int oracle_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     double *o, double *lse,
                     int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk, int64_t D,
                     int causal, double scale, const int64_t *rows, int64_t n_rows) {
    if (Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || Sq < 0 || Sk < 0) return -1;
    if (!rows) n_rows = B * Hq * Sq;
    attention_rows(q, k, v, NULL, 0, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, rows, n_rows);
    return 0;
}

/*
 * Attention evaluated the PASA way in fp64: scores of shifted keys plus the per-block
 * offsets q_i . m_j added back ("global recovering", Abstract). When the shifted keys are
 * exactly k - m_j this equals oracle_attention up to fp64 rounding.
 */
int oracle_attention_recovered(const uint16_t *q, const uint16_t *kshift, const uint16_t *means,
                               int64_t block_rows, const uint16_t *v, double *o, double *lse,
                               int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk,
                               int64_t D, int causal, double scale, const int64_t *rows,
                               int64_t n_rows) {
    if (Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || block_rows <= 0 || !means) return -1;
    if (!rows) n_rows = B * Hq * Sq;
    attention_rows(q, kshift, v, means, block_rows, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale,
                   rows, n_rows);
    return 0;
}

/*
 * Largest |q_i . k_j| over the visible keys of each row, unscaled: the magnitude an fp16
 * score accumulator has to hold. The Abstract names 65504, the largest finite fp16 value,
 * as the overflow threshold.
 */
int oracle_row_max_abs_score(const uint16_t *q, const uint16_t *k, double *out,
                             int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk, int64_t D,
                             int causal, const int64_t *rows, int64_t n_rows) {
    if (Hkv <= 0 || Hq % Hkv != 0 || D <= 0) return -1;
    init_table();
    if (!rows) n_rows = B * Hq * Sq;
    int64_t group = Hq / Hkv;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t g = rows ? rows[r] : r;
        int64_t i = g % Sq;
        int64_t h = (g / Sq) % Hq;
        int64_t b = g / (Sq * Hq);
        const uint16_t *qrow = q + g * D;
        const uint16_t *kh = k + (b * Hkv + h / group) * Sk * D;
        int64_t n = visible_keys(i, Sq, Sk, causal);
        double mx = 0.0;
        for (int64_t j = 0; j < n; ++j) {
            double dot = 0.0;
            for (int64_t d = 0; d < D; ++d) dot += g_h2d[qrow[d]] * g_h2d[kh[j * D + d]];
            if (fabs(dot) > mx) mx = fabs(dot);
        }
        out[r] = mx;
    }
    return 0;
}

/*
 * Largest |q_i . k'_j + q_i . m_(j / block_rows)| over the visible keys of each row, unscaled:
 * the raw score recovered from shifted keys and block means (the quantity PASA's "global
 * recovering" adds back, Abstract). Equals oracle_row_max_abs_score on the raw keys when
 * every shifted key is exactly k - m.
 */
int oracle_row_max_abs_recovered(const uint16_t *q, const uint16_t *kshift, const uint16_t *means,
                                 int64_t block_rows, double *out, int64_t B, int64_t Hq, int64_t Hkv,
                                 int64_t Sq, int64_t Sk, int64_t D, int causal, const int64_t *rows,
                                 int64_t n_rows) {
    if (Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || block_rows <= 0) return -1;
    init_table();
    if (!rows) n_rows = B * Hq * Sq;
    int64_t group = Hq / Hkv;
    int64_t nb = (Sk + block_rows - 1) / block_rows;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t g = rows ? rows[r] : r;
        int64_t i = g % Sq;
        int64_t h = (g / Sq) % Hq;
        int64_t b = g / (Sq * Hq);
        const uint16_t *qrow = q + g * D;
        const uint16_t *kh = kshift + (b * Hkv + h / group) * Sk * D;
        const uint16_t *mh = means + (b * Hkv + h / group) * nb * D;
        int64_t n = visible_keys(i, Sq, Sk, causal);
        double mx = 0.0;
        for (int64_t j = 0; j < n; ++j) {
            double dot = 0.0;
            for (int64_t d = 0; d < D; ++d)
                dot += g_h2d[qrow[d]] * (g_h2d[kh[j * D + d]] + g_h2d[mh[(j / block_rows) * D + d]]);
            if (fabs(dot) > mx) mx = fabs(dot);
        }
        out[r] = mx;
    }
    return 0;
}

/*
 * Per key block, the largest |q_i . k_j| over every query row i and every key j of the
 * block that i sees (causal or not), unscaled: out [B, Hq, ceil(Sk / block_rows)]. A block
 * no row sees gives 0. With k = the shifted keys this is the magnitude the fp16 score
 * accumulator holds for that block; with means != NULL the score is q_i . (k'_j + m_(j /
 * block_rows)), the recovered raw score (Abstract: "global recovering").
 */
int oracle_block_max_abs_score(const uint16_t *q, const uint16_t *k, const uint16_t *means,
                               int64_t block_rows, double *out, int64_t B, int64_t Hq, int64_t Hkv,
                               int64_t Sq, int64_t Sk, int64_t D, int causal) {
    if (Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || block_rows <= 0) return -1;
    init_table();
    int64_t group = Hq / Hkv;
    int64_t nb = (Sk + block_rows - 1) / block_rows;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < B * Hq; ++bh) {
        int64_t b = bh / Hq, h = bh % Hq;
        const uint16_t *kh = k + (b * Hkv + h / group) * Sk * D;
        const uint16_t *mh = means ? means + (b * Hkv + h / group) * nb * D : NULL;
        double *o = out + bh * nb;
        for (int64_t jb = 0; jb < nb; ++jb) o[jb] = 0.0;
        for (int64_t i = 0; i < Sq; ++i) {
            const uint16_t *qrow = q + (bh * Sq + i) * D;
            int64_t n = visible_keys(i, Sq, Sk, causal);
            for (int64_t j = 0; j < n; ++j) {
                double dot = 0.0;
                for (int64_t d = 0; d < D; ++d) {
                    double kv = g_h2d[kh[j * D + d]];
                    if (mh) kv += g_h2d[mh[(j / block_rows) * D + d]];
                    dot += g_h2d[qrow[d]] * kv;
                }
                if (fabs(dot) > o[j / block_rows]) o[j / block_rows] = fabs(dot);
            }
        }
    }
    return 0;
}
