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
int oracle_attn_direct_seg(const void *q, const void *k, const void *v, int dtype,
                           int64_t bs, int64_t L, int hq, int hkv, int hd, double scale, int causal,
                           const int64_t *seg_start, const int64_t *seg_end,
                           const int64_t *rows, int64_t nrows, double *out, double *lse);

int oracle_attn_direct(const void *q, const void *k, const void *v, int dtype,
                       int64_t bs, int64_t L, int hq, int hkv, int hd, double scale, int causal,
                       const int64_t *rows, int64_t nrows, double *out, double *lse)
{
    return oracle_attn_direct_seg(q, k, v, dtype, bs, L, hq, hkv, hd, scale, causal, NULL, NULL, rows, nrows,
                                  out, lse);
}

/*
 * Packed sequences (sequence packing: several samples concatenated into one sequence, each attending
 * only within itself -- the ByteScale motivation on the Context-Parallel page): seg_start[i] and
 * seg_end[i] are the first and one-past-last positions of the sample that position i belongs to.
 * Key j is visible to query i iff seg_start[i] <= j < seg_end[i] and, when causal, j <= i.
 * NULL seg arrays mean one sample spanning the sequence.
 */
int oracle_attn_direct_seg(const void *q, const void *k, const void *v, int dtype,
                           int64_t bs, int64_t L, int hq, int hkv, int hd, double scale, int causal,
                           const int64_t *seg_start, const int64_t *seg_end,
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
                const int64_t j0 = seg_start ? seg_start[i] : 0;
                const int64_t nk = causal ? i + 1 : (seg_end ? seg_end[i] : L);
                for (int d = 0; d < hd; ++d)
                    qi[d] = widen(q, ((b * L + i) * hq + h) * hd + d, dtype);
                double m = -INFINITY;
                for (int64_t j = j0; j < nk; ++j) {
                    const int64_t kb = ((b * L + j) * hkv + kh) * hd;
                    double dot = 0.0;
                    for (int d = 0; d < hd; ++d) dot += qi[d] * widen(k, kb + d, dtype);
                    s[j] = scale * dot;
                    if (s[j] > m) m = s[j];
                }
                double sum = 0.0;
                for (int64_t j = j0; j < nk; ++j) sum += exp(s[j] - m);
                const double l = m + log(sum);
                for (int d = 0; d < hd; ++d) acc[d] = 0.0;
                for (int64_t j = j0; j < nk; ++j) {
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
int oracle_attn_block_seg(const double *q, const int64_t *qpos, const int64_t *qseg, int64_t nq,
                          const double *k, const double *v, const int64_t *kpos, const int64_t *kseg, int64_t nk,
                          int hq, int hkv, int hd, double scale, int causal, double *out, double *lse);

int oracle_attn_block(const double *q, const int64_t *qpos, int64_t nq,
                      const double *k, const double *v, const int64_t *kpos, int64_t nk,
                      int hq, int hkv, int hd, double scale, int causal, double *out, double *lse)
{
    return oracle_attn_block_seg(q, qpos, NULL, nq, k, v, kpos, NULL, nk, hq, hkv, hd, scale, causal, out, lse);
}

/* The same with the sample index of every query and key (packed sequences): key j is kept for query
 * i only if qseg[i] == kseg[j] (and kpos[j] <= qpos[i] when causal); NULL arrays mean one sample. */
int oracle_attn_block_seg(const double *q, const int64_t *qpos, const int64_t *qseg, int64_t nq,
                          const double *k, const double *v, const int64_t *kpos, const int64_t *kseg, int64_t nk,
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
                    keep[j] = (char)((!causal || kpos[j] <= qpos[i]) && (!qseg || qseg[i] == kseg[j]));
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

/*
 * Backward of direct attention: the gradients of the forward above with respect to q, k and v, for
 * an upstream gradient dout of the output (lse is treated as a side result with no gradient).
 * The chain rule through softmax gives, per batch b and query head h (KV head kh = h / G):
 *   P_ij  = exp(s_ij - lse_i)                    (the forward's attention weights, j visible to i)
 *   dP_ij = <dout_i, v_j>
 *   D_i   = sum_j P_ij dP_ij = <dout_i, o_i>
 *   dS_ij = P_ij (dP_ij - D_i)
 *   dq_i  = scale * sum_j dS_ij k_j
 *   dk_j  = scale * sum_{h in the group of kh} sum_i dS_ij q_i
 *   dv_j  = sum_{h in the group of kh} sum_i P_ij dout_i
 * Restricted outputs keep the oracle cheap at long L:
 *   qrows[0..nq): query rows whose dq is returned, dq: (bs, nq, hq, hd) fp64 (nq may be 0);
 *   kv rows j in [j0, L) (j0 = L for none): dk, dv: (bs, L - j0, hkv, hd) fp64. Under the causal
 *   mask only queries i >= j0 see those keys, so only rows [j0, L) need their lse and D; without the
 *   mask every row does.
 * Returns 0, or -1 on a bad argument / allocation failure.
 */
int oracle_attn_bwd_direct_seg(const void *q, const void *k, const void *v, const void *dout, int dtype,
                               int64_t bs, int64_t L, int hq, int hkv, int hd, double scale, int causal,
                               const int64_t *seg_start, const int64_t *seg_end, const int64_t *qrows, int64_t nq,
                               double *dq, int64_t j0, double *dk, double *dv);

int oracle_attn_bwd_direct(const void *q, const void *k, const void *v, const void *dout, int dtype,
                           int64_t bs, int64_t L, int hq, int hkv, int hd, double scale, int causal,
                           const int64_t *qrows, int64_t nq, double *dq, int64_t j0, double *dk, double *dv)
{
    return oracle_attn_bwd_direct_seg(q, k, v, dout, dtype, bs, L, hq, hkv, hd, scale, causal, NULL, NULL, qrows, nq,
                                      dq, j0, dk, dv);
}

/* The same for packed samples (seg_start / seg_end of every position, as oracle_attn_direct_seg):
 * query i and key j interact only inside one sample. */
int oracle_attn_bwd_direct_seg(const void *q, const void *k, const void *v, const void *dout, int dtype,
                               int64_t bs, int64_t L, int hq, int hkv, int hd, double scale, int causal,
                               const int64_t *seg_start, const int64_t *seg_end, const int64_t *qrows, int64_t nq,
                               double *dq, int64_t j0, double *dk, double *dv)
{
    if (bs <= 0 || L <= 0 || hq <= 0 || hkv <= 0 || hd <= 0 || hq % hkv != 0 || nq < 0 || j0 < 0 || j0 > L)
        return -1;
    for (int64_t r = 0; r < nq; ++r)
        if (qrows[r] < 0 || qrows[r] >= L) return -1;
    const int G = hq / hkv;
    const int64_t istat0 = (j0 < L && !causal) ? 0 : j0;  /* rows [istat0, L) feed dk, dv */
    /* per (b, h, i): lse_i and D_i, for the rows that need them */
    char *need = (char *)calloc((size_t)L, 1);
    double *lse = (double *)malloc(sizeof(double) * (size_t)(bs * hq * L));
    double *D = (double *)malloc(sizeof(double) * (size_t)(bs * hq * L));
    if (!need || !lse || !D) {
        free(need); free(lse); free(D);
        return -1;
    }
    for (int64_t r = 0; r < nq; ++r) need[qrows[r]] = 1;
    if (j0 < L)
        for (int64_t i = istat0; i < L; ++i) need[i] = 1;
    int err = 0;

    /* phase 1: forward statistics of every needed row */
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)L);
        double *qi = (double *)malloc(sizeof(double) * (size_t)hd);
        double *o = (double *)malloc(sizeof(double) * (size_t)hd);
        if (!s || !qi || !o) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t t = 0; t < bs * hq * L; ++t) {
                const int64_t i = t % L;
                const int h = (int)((t / L) % hq);
                const int64_t b = t / (L * hq);
                if (!need[i]) continue;
                const int kh = h / G;
                const int64_t ka = seg_start ? seg_start[i] : 0;
                const int64_t nk = causal ? i + 1 : (seg_end ? seg_end[i] : L);
                for (int d = 0; d < hd; ++d) qi[d] = widen(q, ((b * L + i) * hq + h) * hd + d, dtype);
                double m = -INFINITY;
                for (int64_t j = ka; j < nk; ++j) {
                    const int64_t kb = ((b * L + j) * hkv + kh) * hd;
                    double dot = 0.0;
                    for (int d = 0; d < hd; ++d) dot += qi[d] * widen(k, kb + d, dtype);
                    s[j] = scale * dot;
                    if (s[j] > m) m = s[j];
                }
                double sum = 0.0;
                for (int64_t j = ka; j < nk; ++j) sum += exp(s[j] - m);
                const double l = m + log(sum);
                for (int d = 0; d < hd; ++d) o[d] = 0.0;
                for (int64_t j = ka; j < nk; ++j) {
                    const double p = exp(s[j] - l);
                    const int64_t vb = ((b * L + j) * hkv + kh) * hd;
                    for (int d = 0; d < hd; ++d) o[d] += p * widen(v, vb + d, dtype);
                }
                double di = 0.0;
                for (int d = 0; d < hd; ++d) di += widen(dout, ((b * L + i) * hq + h) * hd + d, dtype) * o[d];
                lse[(b * hq + h) * L + i] = l;
                D[(b * hq + h) * L + i] = di;
            }
        }
        free(s); free(qi); free(o);
    }

    /* phase 2: dq of the requested query rows */
    if (!err && nq > 0) {
#pragma omp parallel
        {
            double *qi = (double *)malloc(sizeof(double) * (size_t)hd);
            double *gi = (double *)malloc(sizeof(double) * (size_t)hd);
            double *acc = (double *)malloc(sizeof(double) * (size_t)hd);
            if (!qi || !gi || !acc) {
#pragma omp atomic write
                err = 1;
            } else {
#pragma omp for schedule(dynamic, 4)
                for (int64_t t = 0; t < bs * nq * hq; ++t) {
                    const int h = (int)(t % hq);
                    const int64_t ri = (t / hq) % nq;
                    const int64_t b = t / ((int64_t)hq * nq);
                    const int64_t i = qrows[ri];
                    const int kh = h / G;
                    const int64_t ka = seg_start ? seg_start[i] : 0;
                    const int64_t nk = causal ? i + 1 : (seg_end ? seg_end[i] : L);
                    const double l = lse[(b * hq + h) * L + i], di = D[(b * hq + h) * L + i];
                    for (int d = 0; d < hd; ++d) {
                        qi[d] = widen(q, ((b * L + i) * hq + h) * hd + d, dtype);
                        gi[d] = widen(dout, ((b * L + i) * hq + h) * hd + d, dtype);
                        acc[d] = 0.0;
                    }
                    for (int64_t j = ka; j < nk; ++j) {
                        const int64_t kb = ((b * L + j) * hkv + kh) * hd;
                        double dot = 0.0, dp = 0.0;
                        for (int d = 0; d < hd; ++d) {
                            dot += qi[d] * widen(k, kb + d, dtype);
                            dp += gi[d] * widen(v, kb + d, dtype);
                        }
                        const double p = exp(scale * dot - l);
                        const double ds = p * (dp - di);
                        for (int d = 0; d < hd; ++d) acc[d] += ds * widen(k, kb + d, dtype);
                    }
                    double *o = dq + ((b * nq + ri) * hq + h) * hd;
                    for (int d = 0; d < hd; ++d) o[d] = scale * acc[d];
                }
            }
            free(qi); free(gi); free(acc);
        }
    }

    /* phase 3: dk, dv of key rows [j0, L), summed over the query heads of each KV head */
    if (!err && j0 < L) {
        const int64_t nkv = L - j0;
#pragma omp parallel
        {
            double *kj = (double *)malloc(sizeof(double) * (size_t)hd);
            double *vj = (double *)malloc(sizeof(double) * (size_t)hd);
            double *ak = (double *)malloc(sizeof(double) * (size_t)hd);
            double *av = (double *)malloc(sizeof(double) * (size_t)hd);
            if (!kj || !vj || !ak || !av) {
#pragma omp atomic write
                err = 1;
            } else {
#pragma omp for schedule(dynamic, 4)
                for (int64_t t = 0; t < bs * nkv * hkv; ++t) {
                    const int kh = (int)(t % hkv);
                    const int64_t j = j0 + (t / hkv) % nkv;
                    const int64_t b = t / ((int64_t)hkv * nkv);
                    const int64_t kb = ((b * L + j) * hkv + kh) * hd;
                    for (int d = 0; d < hd; ++d) {
                        kj[d] = widen(k, kb + d, dtype);
                        vj[d] = widen(v, kb + d, dtype);
                        ak[d] = 0.0;
                        av[d] = 0.0;
                    }
                    for (int h = kh * G; h < (kh + 1) * G; ++h) {
                        const int64_t ib = causal ? j : (seg_start ? seg_start[j] : 0);
                        const int64_t ie = seg_end ? seg_end[j] : L;
                        for (int64_t i = ib; i < ie; ++i) {
                            const int64_t qb = ((b * L + i) * hq + h) * hd;
                            double dot = 0.0, dp = 0.0;
                            for (int d = 0; d < hd; ++d) {
                                dot += widen(q, qb + d, dtype) * kj[d];
                                dp += widen(dout, qb + d, dtype) * vj[d];
                            }
                            const double p = exp(scale * dot - lse[(b * hq + h) * L + i]);
                            const double ds = p * (dp - D[(b * hq + h) * L + i]);
                            for (int d = 0; d < hd; ++d) {
                                ak[d] += ds * widen(q, qb + d, dtype);
                                av[d] += p * widen(dout, qb + d, dtype);
                            }
                        }
                    }
                    double *ok = dk + ((b * nkv + (j - j0)) * hkv + kh) * hd;
                    double *ov = dv + ((b * nkv + (j - j0)) * hkv + kh) * hd;
                    for (int d = 0; d < hd; ++d) {
                        ok[d] = scale * ak[d];
                        ov[d] = av[d];
                    }
                }
            }
            free(kj); free(vj); free(ak); free(av);
        }
    }
    free(need); free(lse); free(D);
    return err ? -1 : 0;
}

/*
 * Backward of one ring step's block of attention, accumulated: the contribution of the keys of one
 * KV block to dq of the local queries, and of the local queries to dk, dv of that block. Uses the
 * rows' FINAL lse and D = <dout_i, o_i> of the whole forward (the same formulas as
 * oracle_attn_bwd_direct, restricted to one block; summing the blocks of all ring steps gives the
 * full gradients, because every (query, key) pair belongs to exactly one step).
 *   q, dout: (hq, nq, hd) fp64, qpos[nq], lse, D: (hq, nq)
 *   k, v: (hkv, nk, hd) fp64, kpos[nk]
 *   dq_acc (hq, nq, hd) += ...;  dk_acc, dv_acc (hkv, nk, hd) += ...
 */
int oracle_attn_block_bwd_seg(const double *q, const double *dout, const int64_t *qpos, const int64_t *qseg,
                              const double *lse, const double *D, int64_t nq, const double *k, const double *v,
                              const int64_t *kpos, const int64_t *kseg, int64_t nk, int hq, int hkv, int hd,
                              double scale, int causal, double *dq_acc, double *dk_acc, double *dv_acc);

int oracle_attn_block_bwd(const double *q, const double *dout, const int64_t *qpos, const double *lse,
                          const double *D, int64_t nq, const double *k, const double *v, const int64_t *kpos,
                          int64_t nk, int hq, int hkv, int hd, double scale, int causal, double *dq_acc,
                          double *dk_acc, double *dv_acc)
{
    return oracle_attn_block_bwd_seg(q, dout, qpos, NULL, lse, D, nq, k, v, kpos, NULL, nk, hq, hkv, hd, scale, causal,
                                     dq_acc, dk_acc, dv_acc);
}

/* ... with the sample index of every query and key: pairs from different samples do not interact. */
int oracle_attn_block_bwd_seg(const double *q, const double *dout, const int64_t *qpos, const int64_t *qseg,
                              const double *lse, const double *D, int64_t nq, const double *k, const double *v,
                              const int64_t *kpos, const int64_t *kseg, int64_t nk, int hq, int hkv, int hd,
                              double scale, int causal, double *dq_acc, double *dk_acc, double *dv_acc)
{
    if (nq < 0 || nk < 0 || hq <= 0 || hkv <= 0 || hd <= 0 || hq % hkv != 0) return -1;
    const int G = hq / hkv;
#pragma omp parallel for schedule(dynamic, 8)
    for (int64_t t = 0; t < (int64_t)hq * nq; ++t) {
        const int h = (int)(t / nq);
        const int64_t i = t % nq;
        const int kh = h / G;
        const double *qi = q + ((int64_t)h * nq + i) * hd;
        const double *gi = dout + ((int64_t)h * nq + i) * hd;
        double *acc = dq_acc + ((int64_t)h * nq + i) * hd;
        for (int64_t j = 0; j < nk; ++j) {
            if (causal && kpos[j] > qpos[i]) continue;
            if (qseg && qseg[i] != kseg[j]) continue;
            const double *kj = k + ((int64_t)kh * nk + j) * hd;
            const double *vj = v + ((int64_t)kh * nk + j) * hd;
            double dot = 0.0, dp = 0.0;
            for (int d = 0; d < hd; ++d) {
                dot += qi[d] * kj[d];
                dp += gi[d] * vj[d];
            }
            const double p = exp(scale * dot - lse[(int64_t)h * nq + i]);
            const double ds = p * (dp - D[(int64_t)h * nq + i]);
            for (int d = 0; d < hd; ++d) acc[d] += scale * ds * kj[d];
        }
    }
#pragma omp parallel for schedule(dynamic, 8)
    for (int64_t t = 0; t < (int64_t)hkv * nk; ++t) {
        const int kh = (int)(t / nk);
        const int64_t j = t % nk;
        const double *kj = k + ((int64_t)kh * nk + j) * hd;
        const double *vj = v + ((int64_t)kh * nk + j) * hd;
        double *ak = dk_acc + ((int64_t)kh * nk + j) * hd;
        double *av = dv_acc + ((int64_t)kh * nk + j) * hd;
        for (int h = kh * G; h < (kh + 1) * G; ++h) {
            for (int64_t i = 0; i < nq; ++i) {
                if (causal && kpos[j] > qpos[i]) continue;
                if (qseg && qseg[i] != kseg[j]) continue;
                const double *qi = q + ((int64_t)h * nq + i) * hd;
                const double *gi = dout + ((int64_t)h * nq + i) * hd;
                double dot = 0.0, dp = 0.0;
                for (int d = 0; d < hd; ++d) {
                    dot += qi[d] * kj[d];
                    dp += gi[d] * vj[d];
                }
                const double p = exp(scale * dot - lse[(int64_t)h * nq + i]);
                const double ds = p * (dp - D[(int64_t)h * nq + i]);
                for (int d = 0; d < hd; ++d) {
                    ak[d] += scale * ds * qi[d];
                    av[d] += p * gi[d];
                }
            }
        }
    }
    return 0;
}
