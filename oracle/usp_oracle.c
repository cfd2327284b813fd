/*
 * usp_oracle.c -- TEST INFRASTRUCTURE ONLY: a plain, slow, fp64 CPU reference for the USP-Attention
 * forward path. Only tests/, the package's smoke check and bench.py's CPU-baseline leg may load it.
 * It shares no code, header or constant with the CUDA path.
 *
 * What it computes (the pages' definitions, written out directly):
 *   - softmax attention with its row log-sum-exp, scores s_ij = scale * <q_i, k_j>, causal mask
 *     j <= i on global positions ("Context Parallel 与 Ulysses", section "先弄清楚": each KV block
 *     yields a partial output o_j and lse_j; Fig. 2: the causal mask keeps the lower-left part);
 *       lse_i = m_i + log(sum_j exp(s_ij - m_i)),  m_i = max_j s_ij,
 *       o_i   = sum_j exp(s_ij - lse_i) * v_j;
 *   - the same quantity restricted to one block of keys with explicit global positions, which is
 *     one ring step of LoadBalance-RingAttention (USP review, Algorithm 1 step 4; Context-Parallel
 *     page Fig. 1). A row that sees no key in the block yields (o = 0, lse = -inf), the identity of
 *     the log-sum-exp merge.
 * GQA: query head h reads KV head h / G with G = hq / hkv (contiguous grouping).
 * Arithmetic is fp64 throughout; inputs may be fp32, bf16 (raw 16-bit patterns) or fp64 and are
 * widened exactly. Parallelism is OpenMP over independent rows only: no blocking or reordering of
 * the per-row sums.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_BF16 = 1, OR_F64 = 2 };

static inline double widen(const void *base, int64_t idx, int dtype)
{
    if (dtype == OR_F64) return ((const double *)base)[idx];
    if (dtype == OR_F32) return (double)((const float *)base)[idx];
    /* bf16: the upper 16 bits of an fp32 word; exact widening */
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Direct attention for a list of query rows, natural token order.
 *   q: (bs, L, hq, hd)   k, v: (bs, L, hkv, hd)   (dtype as above)
 *   rows[0..nrows): query positions to evaluate (any order, each in [0, L))
 *   out: (bs, nrows, hq, hd) fp64        lse: (bs, nrows, hq) fp64
 * causal != 0 keeps keys j <= i; otherwise all L keys.
 * Returns 0, or -1 on a bad argument / allocation failure.
 */
int oracle_attn_direct(const void *q, const void *k, const void *v, int dtype,
                       int64_t bs, int64_t L, int hq, int hkv, int hd, double scale, int causal,
                       const int64_t *rows, int64_t nrows, double *out, double *lse)
{
    if (bs <= 0 || L <= 0 || hq <= 0 || hkv <= 0 || hd <= 0 || hq % hkv != 0 || nrows < 0)
        return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= L) return -1;
    const int G = hq / hkv;
    const int64_t ntask = bs * nrows * hq;
    int err = 0;

#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)L);
        double *qi = (double *)malloc(sizeof(double) * (size_t)hd);
        double *acc = (double *)malloc(sizeof(double) * (size_t)hd);
        if (!s || !qi || !acc) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t t = 0; t < ntask; ++t) {
                const int h = (int)(t % hq);
                const int64_t ri = (t / hq) % nrows;
                const int64_t b = t / ((int64_t)hq * nrows);
                const int64_t i = rows[ri];
                const int kh = h / G;
                const int64_t nk = causal ? i + 1 : L;
                for (int d = 0; d < hd; ++d)
                    qi[d] = widen(q, ((b * L + i) * hq + h) * hd + d, dtype);
                double m = -INFINITY;
                for (int64_t j = 0; j < nk; ++j) {
                    const int64_t kb = ((b * L + j) * hkv + kh) * hd;
                    double dot = 0.0;
                    for (int d = 0; d < hd; ++d) dot += qi[d] * widen(k, kb + d, dtype);
                    s[j] = scale * dot;
                    if (s[j] > m) m = s[j];
                }
                double sum = 0.0;
                for (int64_t j = 0; j < nk; ++j) sum += exp(s[j] - m);
                const double l = m + log(sum);
                for (int d = 0; d < hd; ++d) acc[d] = 0.0;
                for (int64_t j = 0; j < nk; ++j) {
                    const double p = exp(s[j] - l);
                    const int64_t vb = ((b * L + j) * hkv + kh) * hd;
                    for (int d = 0; d < hd; ++d) acc[d] += p * widen(v, vb + d, dtype);
                }
                double *o = out + ((b * nrows + ri) * hq + h) * hd;
                for (int d = 0; d < hd; ++d) o[d] = acc[d];
                lse[(b * nrows + ri) * hq + h] = l;
            }
        }
        free(s);
        free(qi);
        free(acc);
    }
    return err ? -1 : 0;
}

/*
 * One block of attention with explicit global positions: the partial (o_j, lse_j) of one ring step.
 *   q: (hq, nq, hd) fp64, qpos[nq]     k, v: (hkv, nk, hd) fp64, kpos[nk]
 *   out: (hq, nq, hd)                  lse: (hq, nq)
 * causal != 0 keeps key j for query i iff kpos[j] <= qpos[i]. Rows with no kept key get
 * o = 0, lse = -inf.
 */
int oracle_attn_block(const double *q, const int64_t *qpos, int64_t nq,
                      const double *k, const double *v, const int64_t *kpos, int64_t nk,
                      int hq, int hkv, int hd, double scale, int causal, double *out, double *lse)
{
    if (nq < 0 || nk < 0 || hq <= 0 || hkv <= 0 || hd <= 0 || hq % hkv != 0) return -1;
    const int G = hq / hkv;
    const int64_t ntask = (int64_t)hq * nq;
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
        char *keep = (char *)malloc((size_t)(nk > 0 ? nk : 1));
        if (!s || !keep) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 8)
            for (int64_t t = 0; t < ntask; ++t) {
                const int h = (int)(t / nq);
                const int64_t i = t % nq;
                const int kh = h / G;
                const double *qi = q + ((int64_t)h * nq + i) * hd;
                double m = -INFINITY;
                int64_t nkeep = 0;
                for (int64_t j = 0; j < nk; ++j) {
                    keep[j] = (char)(!causal || kpos[j] <= qpos[i]);
                    if (!keep[j]) continue;
                    ++nkeep;
                    const double *kj = k + ((int64_t)kh * nk + j) * hd;
                    double dot = 0.0;
                    for (int d = 0; d < hd; ++d) dot += qi[d] * kj[d];
                    s[j] = scale * dot;
                    if (s[j] > m) m = s[j];
                }
                double *o = out + ((int64_t)h * nq + i) * hd;
                if (nkeep == 0) {
                    for (int d = 0; d < hd; ++d) o[d] = 0.0;
                    lse[(int64_t)h * nq + i] = -INFINITY;
                    continue;
                }
                double sum = 0.0;
                for (int64_t j = 0; j < nk; ++j)
                    if (keep[j]) sum += exp(s[j] - m);
                const double l = m + log(sum);
                for (int d = 0; d < hd; ++d) o[d] = 0.0;
                for (int64_t j = 0; j < nk; ++j) {
                    if (!keep[j]) continue;
                    const double p = exp(s[j] - l);
                    const double *vj = v + ((int64_t)kh * nk + j) * hd;
                    for (int d = 0; d < hd; ++d) o[d] += p * vj[d];
                }
                lse[(int64_t)h * nq + i] = l;
            }
        }
        free(s);
        free(keep);
    }
    return err ? -1 : 0;
}
