/*
 * attn_ref.c -- plain fp64 CPU oracle for the attention forward and backward passes.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file.  Its only users are the tests, the smoke check and the CPU
 * baseline / reference arm of the benchmark.  It shares no code, header,
 * table or helper with the CUDA path.
 *
 * Sources (page titles as printed on the pages):
 *   [GKFA]  "GPU 内核与 FlashAttention" (hs-black, scaling-gpu-kernels)
 *             §10   standard attention: S = Q K^T (times the scale), P = softmax(S), O = P V
 *             §11.1 safe softmax: subtract the row maximum before exp
 *             §11.2 merge of two partial (m, l) pairs
 *             §11.3 online output recurrence (m, l, o-tilde), o = o-tilde / l
 *             §13.2 and §14.1 the forward keeps only L = m + log l per row
 *   [FMHA] "Flash Attention实现深度解析" (maplevalley) §3.1: the host entry
 *             returns {out, softmax_lse} with lse shaped [batch, heads, max_seqlen_q]
 *   [CH2]  "Flash Attention 2 Chapter2": tensors are [batch, seq, heads, d_head]
 *             (the generate_qkv listing in the section on mapping tensors to mma)
 *
 * Definition computed here (all arithmetic in double, on the bf16 input values
 * widened exactly):
 *   s_ij  = scale * sum_c q_ic k_jc                      ([GKFA] §10)
 *   m_i   = max_j s_ij                                   ([GKFA] §11.1)
 *   p_ij  = exp(s_ij - m_i),  l_i = sum_j p_ij,  P_ij = p_ij / l_i
 *   o_ic  = sum_j P_ij v_jc                              ([GKFA] §10)
 *   LSE_i = m_i + ln(l_i)   (natural log, scaled-score units; [GKFA] §13.2)
 * The full S row block of one (batch, head) is materialised, then turned into
 * P in place, then multiplied by V: no blocking, no fusion.
 *
 * Rows that have no key at all (an empty key sequence, or a causal row that
 * sees no key) have no softmax.  The pages are silent; this oracle returns
 * o = 0 and LSE = -inf for them (log of an empty sum).
 *
 * Causal masking ([GKFA] §14.4): scores with key index j > i are -inf.  When
 * the query and key lengths differ the pages are silent; this oracle aligns
 * the mask bottom-right, i.e. query i sees keys j <= i + (Nk - Nq), which is
 * j <= i for equal lengths.
 *
 * Grouped key/value heads ([GKFA] §14.2, MQA/GQA): with Hk key/value heads and
 * H = G * Hk query heads, query head h reads key/value head h / G.
 *
 * Backward pass ([GKFA] §13.1), oracle_attn_bwd_dense(): for a loss phi with
 * dO = d phi / d O given, and P the full softmax above (materialised),
 *   dV = P^T dO
 *   dP = dO V^T                       (dP_ij = do_i . v_j)
 *   D_i = sum_j P_ij dP_ij            (the definition; §13.1 shows D_i = do_i . o_i)
 *   dS = P o (dP - D)                 (softmax Jacobian, row by row)
 *   dQ = scale * dS K,  dK = scale * dS^T Q
 * The factor scale appears because S = scale * Q K^T.  With grouped heads the
 * key/value gradients of the G query heads that share a K/V head are summed
 * ([GKFA] §14.2).  Rows that see no key have P = 0 and contribute nothing.
 *
 * FP8 ([GKFA] §15.5, block quantisation), oracle_attn_fp8_dense(): the inputs
 * are e4m3 codes with fp32 scales; each value is decoded from the e4m3 format
 * definition (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
 * exponent field 0 is subnormal, m/8 * 2^-6; code 0x7f/0xff is NaN; no
 * infinities) and multiplied by its block scale, and the definition above is
 * evaluated on those values in double.  oracle_e4m3_encode() is the nearest
 * code (ties to the even mantissa, saturating to +-448), found by comparing
 * against every finite code: the reference for the quantiser.
 *
 * oracle_attn_online() restates the blockwise recurrence of [GKFA] §11.3 with
 * the deferred division of §14.1, again in double.  It exists only so tests can
 * check the pages' claim that the recurrence is exact (it must agree with the
 * full definition to rounding).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_double(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * One head: nq query rows against nk key/value rows.
 *   q row i  starts at q + i * q_rs     (d elements, contiguous)
 *   k/v row j starts at k/v + j * kv_rs
 *   o row i  starts at o + i * o_rs     (d doubles)
 *   lse of row i at lse[i * lse_stride]
 * Returns 0, or -1 when the S block cannot be allocated.
 */
static int head_attention(const uint16_t *q, size_t q_rs, int nq,
                          const uint16_t *k, const uint16_t *v, size_t kv_rs, int nk,
                          int d, double scale, int causal, long row0, long offset,
                          double *o, size_t o_rs, double *lse, size_t lse_stride)
{
    if (nq <= 0)
        return 0;
    if (nk <= 0) {
        for (int i = 0; i < nq; ++i) {
            for (int c = 0; c < d; ++c)
                o[(size_t)i * o_rs + c] = 0.0;
            lse[(size_t)i * lse_stride] = -INFINITY;
        }
        return 0;
    }
    double *S = (double *)malloc((size_t)nq * (size_t)nk * sizeof(double));
    if (!S)
        return -1;

    /* S = scale * Q K^T, materialised ([GKFA] §10).  Under the causal mask,
       row i (absolute index row0 + i) sees keys j <= row0 + i + offset only;
       the others are -inf ([GKFA] §14.4). */
    for (int i = 0; i < nq; ++i) {
        const uint16_t *qi = q + (size_t)i * q_rs;
        for (int j = 0; j < nk; ++j) {
            if (causal && (long)j > row0 + i + offset) {
                S[(size_t)i * nk + j] = -INFINITY;
                continue;
            }
            const uint16_t *kj = k + (size_t)j * kv_rs;
            double acc = 0.0;
            for (int c = 0; c < d; ++c)
                acc += bf16_to_double(qi[c]) * bf16_to_double(kj[c]);
            S[(size_t)i * nk + j] = scale * acc;
        }
    }

    /* Safe softmax, row by row, three passes: max, exp and sum, divide
       ([GKFA] §11.1).  P overwrites S.  A row whose scores are all -inf has
       no softmax: o = 0, LSE = -inf. */
    for (int i = 0; i < nq; ++i) {
        double *row = S + (size_t)i * nk;
        double m = row[0];
        for (int j = 1; j < nk; ++j)
            if (row[j] > m)
                m = row[j];
        if (m == -INFINITY) {
            for (int j = 0; j < nk; ++j)
                row[j] = 0.0;
            lse[(size_t)i * lse_stride] = -INFINITY;
            continue;
        }
        double l = 0.0;
        for (int j = 0; j < nk; ++j) {
            row[j] = exp(row[j] - m);
            l += row[j];
        }
        for (int j = 0; j < nk; ++j)
            row[j] /= l;
        lse[(size_t)i * lse_stride] = m + log(l); /* [GKFA] §13.2 */
    }

    /* O = P V ([GKFA] §10). */
    for (int i = 0; i < nq; ++i) {
        const double *prow = S + (size_t)i * nk;
        double *oi = o + (size_t)i * o_rs;
        for (int c = 0; c < d; ++c)
            oi[c] = 0.0;
        for (int j = 0; j < nk; ++j) {
            const uint16_t *vj = v + (size_t)j * kv_rs;
            const double p = prow[j];
            for (int c = 0; c < d; ++c)
                oi[c] += p * bf16_to_double(vj[c]);
        }
    }
    free(S);
    return 0;
}

/*
 * Backward of one head (definitions in the header comment).  q/do rows i at
 * q + i*q_rs and dout + i*q_rs; k/v rows j at k + j*kv_rs.  dq row i is
 * written at dq + i*q_rs; dk/dv row j is ADDED at dk/dv + j*kv_rs (doubles),
 * so query heads sharing a key/value head accumulate.  delta[i*delta_stride]
 * receives D_i.  Returns 0, or -1 when P cannot be allocated.
 */
static int head_attention_bwd(const uint16_t *q, const uint16_t *dout, size_t q_rs, int nq,
                              const uint16_t *k, const uint16_t *v, size_t kv_rs, int nk,
                              int d, double scale, int causal, long offset,
                              double *dq, double *dk, double *dv, double *delta,
                              size_t delta_stride)
{
    if (nq <= 0)
        return 0;
    double *P = (double *)malloc((size_t)nq * (size_t)(nk > 0 ? nk : 1) * sizeof(double));
    double *dP = (double *)malloc((size_t)nq * (size_t)(nk > 0 ? nk : 1) * sizeof(double));
    if (!P || !dP) {
        free(P);
        free(dP);
        return -1;
    }
    /* P: the forward's softmax, materialised (S = scale Q K^T, causal -inf,
       safe softmax, rows with no visible key all zero). */
    for (int i = 0; i < nq; ++i) {
        double *row = P + (size_t)i * nk;
        double m = -INFINITY;
        for (int j = 0; j < nk; ++j) {
            if (causal && (long)j > i + offset) {
                row[j] = -INFINITY;
                continue;
            }
            double acc = 0.0;
            for (int c = 0; c < d; ++c)
                acc += bf16_to_double(q[(size_t)i * q_rs + c]) * bf16_to_double(k[(size_t)j * kv_rs + c]);
            row[j] = scale * acc;
            if (row[j] > m)
                m = row[j];
        }
        double l = 0.0;
        for (int j = 0; j < nk; ++j) {
            row[j] = (m == -INFINITY) ? 0.0 : exp(row[j] - m);
            l += row[j];
        }
        for (int j = 0; j < nk; ++j)
            row[j] = (l > 0.0) ? row[j] / l : 0.0;
    }
    /* dV += P^T dO. */
    for (int j = 0; j < nk; ++j) {
        double *dvj = dv + (size_t)j * kv_rs;
        for (int i = 0; i < nq; ++i) {
            const double pij = P[(size_t)i * nk + j];
            if (pij == 0.0)
                continue;
            for (int c = 0; c < d; ++c)
                dvj[c] += pij * bf16_to_double(dout[(size_t)i * q_rs + c]);
        }
    }
    /* dP = dO V^T; D_i = sum_j P_ij dP_ij; dS = P o (dP - D), stored over dP. */
    for (int i = 0; i < nq; ++i) {
        double Di = 0.0;
        for (int j = 0; j < nk; ++j) {
            double acc = 0.0;
            for (int c = 0; c < d; ++c)
                acc += bf16_to_double(dout[(size_t)i * q_rs + c]) * bf16_to_double(v[(size_t)j * kv_rs + c]);
            dP[(size_t)i * nk + j] = acc;
            Di += P[(size_t)i * nk + j] * acc;
        }
        delta[(size_t)i * delta_stride] = Di;
        for (int j = 0; j < nk; ++j)
            dP[(size_t)i * nk + j] = P[(size_t)i * nk + j] * (dP[(size_t)i * nk + j] - Di);
    }
    /* dQ = scale dS K;  dK += scale dS^T Q. */
    for (int i = 0; i < nq; ++i) {
        double *dqi = dq + (size_t)i * q_rs;
        for (int c = 0; c < d; ++c)
            dqi[c] = 0.0;
        for (int j = 0; j < nk; ++j) {
            const double ds = dP[(size_t)i * nk + j];
            if (ds == 0.0)
                continue;
            for (int c = 0; c < d; ++c)
                dqi[c] += scale * ds * bf16_to_double(k[(size_t)j * kv_rs + c]);
        }
    }
    for (int j = 0; j < nk; ++j) {
        double *dkj = dk + (size_t)j * kv_rs;
        for (int i = 0; i < nq; ++i) {
            const double ds = dP[(size_t)i * nk + j];
            if (ds == 0.0)
                continue;
            for (int c = 0; c < d; ++c)
                dkj[c] += scale * ds * bf16_to_double(q[(size_t)i * q_rs + c]);
        }
    }
    free(P);
    free(dP);
    return 0;
}

/*
 * Dense backward.  q, dout, dq: [B, Nq, H, d]; k, v, dk, dv: [B, Nk, Hk, d];
 * delta: [B, H, Nq] (D_i).  Inputs are bf16 bit patterns, outputs double.
 * Parallel over (b, key/value head); the G query heads of a group run in
 * order inside one task, so their dK/dV sums need no atomics.
 */
int oracle_attn_bwd_dense(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          const uint16_t *dout, int B, int Nq, int Nk, int H, int Hk, int d,
                          double scale, int causal, double *dq, double *dk, double *dv,
                          double *delta)
{
    if (Hk <= 0 || H % Hk != 0)
        return -1;
    int err = 0;
    const int G = H / Hk;
    const size_t q_rs = (size_t)H * d, kv_rs = (size_t)Hk * d;
#pragma omp parallel for collapse(2) schedule(dynamic, 1) reduction(| : err)
    for (int b = 0; b < B; ++b) {
        for (int hk = 0; hk < Hk; ++hk) {
            const size_t kvoff = (size_t)b * Nk * Hk * d + (size_t)hk * d;
            for (int j = 0; j < Nk; ++j)
                for (int c = 0; c < d; ++c) {
                    dk[kvoff + (size_t)j * kv_rs + c] = 0.0;
                    dv[kvoff + (size_t)j * kv_rs + c] = 0.0;
                }
            for (int g = 0; g < G; ++g) {
                const int h = hk * G + g;
                const size_t qoff = (size_t)b * Nq * H * d + (size_t)h * d;
                err |= head_attention_bwd(q + qoff, dout + qoff, q_rs, Nq, k + kvoff, v + kvoff,
                                          kv_rs, Nk, d, scale, causal, (long)Nk - Nq, dq + qoff,
                                          dk + kvoff, dv + kvoff,
                                          delta + ((size_t)b * H + h) * Nq, 1);
            }
        }
    }
    return err ? -1 : 0;
}

/* e4m3 code -> value (NaN for 0x7f / 0xff). */
double oracle_e4m3_decode(uint8_t c)
{
    const int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7)
        return NAN;
    const double mag = (e == 0) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* Nearest e4m3 code to x: round to nearest, ties to the even mantissa,
   saturating to the largest finite magnitude (448); NaN -> 0x7f. */
uint8_t oracle_e4m3_encode(double x)
{
    if (x != x)
        return 0x7f;
    const int neg = x < 0 || (x == 0 && signbit(x));
    const double a = fabs(x);
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c <= 0x7e; ++c) {
        const double v = oracle_e4m3_decode((uint8_t)c);
        const double dd = fabs(v - a);
        if (dd < best_d || (dd == best_d && (c & 1) == 0 && (best & 1) == 1)) {
            best_d = dd;
            best = c;
        }
    }
    if (a >= 448.0)
        best = 0x7e;
    return (uint8_t)(best | (neg ? 0x80 : 0));
}

/* codes[i] = nearest code to x[i] / scale, the division done in float. */
void oracle_quantize_e4m3(const float *x, long long n, float scale, uint8_t *codes)
{
    for (long long i = 0; i < n; ++i) {
        const float y = x[i] / scale;
        codes[i] = oracle_e4m3_encode((double)y);
    }
}

/* One head in double: nq query rows (q row i at q + i * d), nk keys (k row j
   at k + j * d, v row j at v + j * d); o row i at o + i * o_rs.  Optional
   outputs (NULL: not computed): mrow[i] = max_j s_ij over the keys row i sees
   (-inf if none), and abs_o row i (at abs_o + i * o_rs) = sum_j P_ij |v_j|,
   the same weights applied to the magnitudes of V. */
static int head_attention_f64(const double *q, int nq, const double *k, const double *v, int nk, int d,
                              double scale, int causal, long offset, double *o, size_t o_rs,
                              double *lse, double *mrow, double *abs_o)
{
    double *S = (double *)malloc((size_t)(nq > 0 ? nq : 1) * (size_t)(nk > 0 ? nk : 1) * sizeof(double));
    if (!S)
        return -1;
    for (int i = 0; i < nq; ++i) {
        double *row = S + (size_t)i * nk;
        double m = -INFINITY;
        for (int j = 0; j < nk; ++j) {
            if (causal && (long)j > i + offset) {
                row[j] = -INFINITY;
                continue;
            }
            double acc = 0.0;
            for (int c = 0; c < d; ++c)
                acc += q[(size_t)i * d + c] * k[(size_t)j * d + c];
            row[j] = scale * acc;
            if (row[j] > m)
                m = row[j];
        }
        double *oi = o + (size_t)i * o_rs;
        double *ai = abs_o ? abs_o + (size_t)i * o_rs : NULL;
        for (int c = 0; c < d; ++c)
            oi[c] = 0.0;
        if (ai)
            for (int c = 0; c < d; ++c)
                ai[c] = 0.0;
        if (mrow)
            mrow[i] = m;
        if (m == -INFINITY) {
            lse[i] = -INFINITY;
            continue;
        }
        double l = 0.0;
        for (int j = 0; j < nk; ++j) {
            row[j] = exp(row[j] - m);
            l += row[j];
        }
        for (int j = 0; j < nk; ++j) {
            const double pj = row[j] / l;
            for (int c = 0; c < d; ++c)
                oi[c] += pj * v[(size_t)j * d + c];
            if (ai)
                for (int c = 0; c < d; ++c)
                    ai[c] += pj * fabs(v[(size_t)j * d + c]);
        }
        lse[i] = m + log(l);
    }
    free(S);
    return 0;
}

/*
 * FP8 dense form.  q8: [B, Nq, H, d] codes, k8: [B, Nk, Hk, d], vt8: [B, Hk, d,
 * nk_pad] (V transposed); q_scale [B, H, ceil(Nq/128)], k_scale [B, Hk,
 * ceil(Nk/128)], v_scale [B, Hk].  o: [B, Nq, H, d], lse: [B, H, Nq] (double).
 * Optional (NULL: skipped): rowmax [B, H, Nq], the largest score each row sees,
 * and abs_o [B, Nq, H, d], sum_j P_ij |v_j| -- the two plain quantities that
 * bound the effect of rounding the weights P to e4m3 (tests only).
 */
int oracle_attn_fp8_dense(const uint8_t *q8, const uint8_t *k8, const uint8_t *vt8, const float *q_scale,
                          const float *k_scale, const float *v_scale, int B, int Nq, int Nk, int H, int Hk,
                          int d, int nk_pad, double scale, int causal, double *o, double *lse,
                          double *rowmax, double *abs_o)
{
    if (Hk <= 0 || H % Hk != 0)
        return -1;
    const int G = H / Hk, qb = (Nq + 127) / 128, kb = (Nk + 127) / 128;
    int err = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1) reduction(| : err)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            const int hk = h / G;
            double *q = (double *)malloc((size_t)(Nq > 0 ? Nq : 1) * d * sizeof(double));
            double *k = (double *)malloc((size_t)(Nk > 0 ? Nk : 1) * d * sizeof(double));
            double *v = (double *)malloc((size_t)(Nk > 0 ? Nk : 1) * d * sizeof(double));
            if (!q || !k || !v) {
                free(q); free(k); free(v);
                err |= 1;
                continue;
            }
            for (int i = 0; i < Nq; ++i)
                for (int c = 0; c < d; ++c)
                    q[(size_t)i * d + c] = oracle_e4m3_decode(q8[(((size_t)b * Nq + i) * H + h) * d + c]) *
                                           (double)q_scale[((size_t)b * H + h) * qb + i / 128];
            for (int j = 0; j < Nk; ++j)
                for (int c = 0; c < d; ++c) {
                    k[(size_t)j * d + c] = oracle_e4m3_decode(k8[(((size_t)b * Nk + j) * Hk + hk) * d + c]) *
                                           (double)k_scale[((size_t)b * Hk + hk) * kb + j / 128];
                    v[(size_t)j * d + c] = oracle_e4m3_decode(vt8[(((size_t)b * Hk + hk) * d + c) * nk_pad + j]) *
                                           (double)v_scale[(size_t)b * Hk + hk];
                }
            err |= head_attention_f64(q, Nq, k, v, Nk, d, scale, causal, (long)Nk - Nq,
                                      o + (size_t)b * Nq * H * d + (size_t)h * d, (size_t)H * d,
                                      lse + ((size_t)b * H + h) * Nq,
                                      rowmax ? rowmax + ((size_t)b * H + h) * Nq : NULL,
                                      abs_o ? abs_o + (size_t)b * Nq * H * d + (size_t)h * d : NULL);
            free(q); free(k); free(v);
        }
    }
    return err ? -1 : 0;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * Dense form.  q, o: [B, Nq, H, d]; k, v: [B, Nk, Hk, d]; lse: [B, H, Nq].
 * Inputs are bf16 bit patterns; outputs are double.
 * Parallel over (b, h) only.  Returns 0, or -1 on allocation failure.
 */
int oracle_attn_dense(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      int B, int Nq, int Nk, int H, int Hk, int d, double scale, int causal,
                      double *o, double *lse)
{
    if (Hk <= 0 || H % Hk != 0)
        return -1;
    int err = 0;
    const int G = H / Hk;
    const size_t q_rs = (size_t)H * d, kv_rs = (size_t)Hk * d;
#pragma omp parallel for collapse(2) schedule(dynamic, 1) reduction(| : err)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            const size_t qoff = (size_t)b * Nq * H * d + (size_t)h * d;
            const size_t kvoff = (size_t)b * Nk * Hk * d + (size_t)(h / G) * d;
            err |= head_attention(q + qoff, q_rs, Nq, k + kvoff, v + kvoff, kv_rs, Nk, d, scale,
                                  causal, 0, (long)Nk - Nq,
                                  o + qoff, q_rs, lse + ((size_t)b * H + h) * Nq, 1);
        }
    }
    return err ? -1 : 0;
}

/*
 * Selected rows of the dense form: rows[3*r .. 3*r+2] = (b, h, i).
 * o_rows: [n_rows, d]; lse_rows: [n_rows].  Each row is computed with the
 * same per-head routine as oracle_attn_dense (a one-row head).
 */
int oracle_attn_dense_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                           int B, int Nq, int Nk, int H, int Hk, int d, double scale, int causal,
                           int n_rows, const int64_t *rows, double *o_rows, double *lse_rows)
{
    if (Hk <= 0 || H % Hk != 0)
        return -1;
    int err = 0;
    const int G = H / Hk;
    const size_t kv_rs = (size_t)Hk * d;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int r = 0; r < n_rows; ++r) {
        const int64_t b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
        if (b < 0 || b >= B || h < 0 || h >= H || i < 0 || i >= Nq) {
            err |= 1;
            continue;
        }
        const size_t qoff = (((size_t)b * Nq + i) * H + h) * d;
        const size_t kvoff = (size_t)b * Nk * Hk * d + (size_t)(h / G) * d;
        err |= head_attention(q + qoff, 0, 1, k + kvoff, v + kvoff, kv_rs, Nk, d, scale,
                              causal, (long)i, (long)Nk - Nq,
                              o_rows + (size_t)r * d, 0, lse_rows + r, 1);
    }
    return err ? -1 : 0;
}

/*
 * Variable-length packed form ([FMHA] §3.1).  Sequence b owns query rows
 * [cu_q[b], cu_q[b+1]) and key rows [cu_k[b], cu_k[b+1]) of the packed
 * tensors q, o: [total_q, H, d] and k, v: [total_k, Hk, d].  Each sequence
 * attends only within itself.  lse: [B, H, max_seqlen_q]; entry
 * (b, h, i) is written for i < len_q(b) only.
 */
int oracle_attn_varlen(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       const int32_t *cu_q, const int32_t *cu_k, int B, int H, int Hk, int d,
                       double scale, int causal, int max_seqlen_q, double *o, double *lse)
{
    if (Hk <= 0 || H % Hk != 0)
        return -1;
    int err = 0;
    const int G = H / Hk;
    const size_t rs = (size_t)H * d, kv_rs = (size_t)Hk * d;
#pragma omp parallel for collapse(2) schedule(dynamic, 1) reduction(| : err)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            const int nq = cu_q[b + 1] - cu_q[b];
            const int nk = cu_k[b + 1] - cu_k[b];
            if (nq > max_seqlen_q) {
                err |= 1;
                continue;
            }
            const size_t qoff = (size_t)cu_q[b] * rs + (size_t)h * d;
            const size_t kvoff = (size_t)cu_k[b] * kv_rs + (size_t)(h / G) * d;
            err |= head_attention(q + qoff, rs, nq, k + kvoff, v + kvoff, kv_rs, nk, d, scale,
                                  causal, 0, (long)nk - nq,
                                  o + qoff, rs, lse + ((size_t)b * H + h) * max_seqlen_q, 1);
        }
    }
    return err ? -1 : 0;
}

/*
 * Blockwise online recurrence, dense form, in double ([GKFA] §11.3, §14.1).
 * For each query row keep m (running max), l (running sum) and the
 * unnormalised output o~.  For each block of `block` keys:
 *   m'  = max(m, max_j s_j)
 *   l   = e^(m - m') l  + sum_j e^(s_j - m')
 *   o~  = e^(m - m') o~ + sum_j e^(s_j - m') v_j
 *   m   = m'
 * After the last block: o = o~ / l and LSE = m + ln l.
 * Start values: m = -inf, l = 0, o~ = 0 (first correction factor e^-inf = 0).
 */
int oracle_attn_online(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       int B, int Nq, int Nk, int H, int d, double scale, int block,
                       double *o, double *lse)
{
    if (block <= 0)
        return -1;
    int err = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1) reduction(| : err)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            double *ot = (double *)malloc((size_t)d * sizeof(double));
            double *s = (double *)malloc((size_t)block * sizeof(double));
            if (!ot || !s) {
                free(ot);
                free(s);
                err |= 1;
                continue;
            }
            for (int i = 0; i < Nq; ++i) {
                const uint16_t *qi = q + (((size_t)b * Nq + i) * H + h) * d;
                double m = -INFINITY, l = 0.0;
                for (int c = 0; c < d; ++c)
                    ot[c] = 0.0;
                for (int j0 = 0; j0 < Nk; j0 += block) {
                    const int nb = (Nk - j0 < block) ? (Nk - j0) : block;
                    double bmax = -INFINITY;
                    for (int jj = 0; jj < nb; ++jj) {
                        const uint16_t *kj = k + (((size_t)b * Nk + j0 + jj) * H + h) * d;
                        double acc = 0.0;
                        for (int c = 0; c < d; ++c)
                            acc += bf16_to_double(qi[c]) * bf16_to_double(kj[c]);
                        s[jj] = scale * acc;
                        if (s[jj] > bmax)
                            bmax = s[jj];
                    }
                    const double mn = (bmax > m) ? bmax : m;
                    const double corr = exp(m - mn); /* 0 on the first block */
                    l *= corr;
                    for (int c = 0; c < d; ++c)
                        ot[c] *= corr;
                    for (int jj = 0; jj < nb; ++jj) {
                        const double p = exp(s[jj] - mn);
                        const uint16_t *vj = v + (((size_t)b * Nk + j0 + jj) * H + h) * d;
                        l += p;
                        for (int c = 0; c < d; ++c)
                            ot[c] += p * bf16_to_double(vj[c]);
                    }
                    m = mn;
                }
                double *oi = o + (((size_t)b * Nq + i) * H + h) * d;
                if (Nk <= 0) {
                    for (int c = 0; c < d; ++c)
                        oi[c] = 0.0;
                    lse[((size_t)b * H + h) * Nq + i] = -INFINITY;
                } else {
                    for (int c = 0; c < d; ++c)
                        oi[c] = ot[c] / l;
                    lse[((size_t)b * H + h) * Nq + i] = m + log(l);
                }
            }
            free(ot);
            free(s);
        }
    }
    return err ? -1 : 0;
}
