/*
 * attention_oracle.c -- plain fp64 CPU oracle for exact softmax attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header or table with the CUDA
 * kernels of the library.
 *
 * What it computes is the plain definition of attention, not the tiled
 * algorithm.  The tiled method reaches the same numbers up to rounding order
 * ("exact attention": FlashAttention: exact attention made fast by counting
 * memory traffic, "The method"; FlashAttention and IO-aware exact attention,
 * "Common misconceptions").  So the oracle is the definition written out:
 *
 *   s_ij  = scale * sum_c q_ic k_jc, and s_ij = -inf when causal and j > i
 *           (Flash Attention, "The Memory Wall Problem", step 1: S = Q K^T;
 *            the scale and the causal rule are the library's documented
 *            reading of an argument the pages leave open)
 *   m_i   = max_j s_ij,  e_ij = exp(s_ij - m_i),  l_i = sum_j e_ij,
 *   p_ij  = e_ij / l_i
 *           (Flash Attention, "Online Softmax Algorithm", safe softmax)
 *   o_ic  = sum_j p_ij v_jc
 *           (Flash Attention, "The Memory Wall Problem", step 3: O = P V)
 *   lse_i = m_i + log(l_i)   -- natural log of sum_j exp(s_ij)
 *           (FlashAttention and IO-aware exact attention, "Core ideas":
 *            one log-sum-exp per row is what the forward keeps)
 *
 * Backward, for a loss L with dL/dO = dO given.  The pages say the backward
 * recomputes P from Q, K, V and the row statistics (paper review, "The
 * method"; "Backward by recomputation" in the curriculum note) but print no
 * gradient formulas; these are the chain rule through the three steps above
 * (softmax Jacobian), pinned in the tests by finite differences:
 *
 *   dv_jc = sum_i p_ij dO_ic
 *   dp_ij = sum_c dO_ic v_jc
 *   D_i   = sum_j p_ij dp_ij          (equal to sum_c dO_ic o_ic)
 *   ds_ij = p_ij (dp_ij - D_i)
 *   dq_ic = scale * sum_j ds_ij k_jc
 *   dk_jc = scale * sum_i ds_ij q_ic
 *
 * Grouped key/value heads (GQA; MQA when there is one key/value head): the
 * pages note that FlashAttention 2 and 3 support multi-query and
 * grouped-query attention (Flash Attention, "Evolution: Flash Attention 2 &
 * 3") without defining the grouping.  Reading taken: with BH query heads and
 * BH / G key/value heads, query head h attends with key/value head h / G
 * (integer division; G consecutive query heads share one K, V).  By the
 * chain rule through the shared K and V, dk and dv of key/value head hk sum
 * the per-head terms above over its query heads hk*G ... hk*G + G - 1.
 *
 * Query and key lengths may differ (Nq query rows, Nk keys; the pages list
 * variable sequence lengths among FlashAttention 2's changes, Flash
 * Attention, "Evolution: Flash Attention 2 & 3").  Causal masking then
 * aligns the last query with the last key (the library's reading): key j is
 * visible to query i iff j <= i + (Nk - Nq), which is j <= i when the
 * lengths are equal; it requires Nk >= Nq so that every row sees a key.
 *
 * Block-sparse attention: the pages name a block-sparse extension of the
 * method (FlashAttention: exact attention made fast by counting memory
 * traffic, "The method", Sec 3.3) and list predefined block-sparse patterns
 * among the sparse variants (Flash Attention, "Sparse Flash Attention"),
 * without giving their form.  Reading taken: an optional block mask
 * bm[ceil(Nq/bq)][ceil(Nk/bk)] (row-major, shared by every head) marks which
 * bq x bk blocks of (query rows, keys) are kept; key j is visible to query i
 * only if bm[i/bq][j/bk] != 0, on top of the causal rule.  A row that sees
 * no key at all has an empty sum: l_i = 0, so lse_i = -inf, o_i = 0, and it
 * contributes nothing to any gradient (dq_i = 0, D_i = 0).
 *
 * Layout: every tensor is a dense fp64 array [heads][rows][d] (d innermost);
 * q, o, dO, dq have BH heads of Nq rows, k, v, dk, dv BH / G heads of Nk
 * rows; lse and the per-row statistics are [BH][Nq].  BH = B*H independent
 * query heads.
 * oracle_attn_fwd_rows and oracle_attn_bwd_rows compute the same formulas
 * for chosen rows of one head (sampled checks of long sequences).
 * Parallelism: OpenMP over (head, row) for the row-wise passes and over
 * (head, key) for the key-wise pass.  No blocking, no online softmax, no
 * reordering beyond the loops of the definition.
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* number of threads the oracle will use (for reporting) */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Which keys a query sees: the causal rule (off = Nk - Nq >= 0) and the
 * optional block mask (bm == NULL: every block kept). */
typedef struct {
    int causal;
    long off;
    const unsigned char *bm;
    int bq, bk, nbk; /* block sizes; blocks per mask row */
} Mask;

/* key j is visible to query i: j <= i + off when causal, and its block kept */
static int visible(const Mask *mk, long i, long j) {
    if (mk->causal && j > i + mk->off) return 0;
    return !mk->bm || mk->bm[(i / mk->bq) * (long)mk->nbk + j / mk->bk] != 0;
}

/* s_ij = scale * q_i . k_j (no masking here; callers skip invisible keys) */
static double score(const double *qi, const double *kj, int d, double scale) {
    double acc = 0.0;
    for (int c = 0; c < d; ++c) acc += qi[c] * kj[c];
    return scale * acc;
}

/* Row statistics of the safe softmax of row i: m_i and l_i. */
static void row_stats(const double *q, const double *k, long i, int Nk, const Mask *mk, int d,
                      double scale, double *m_out, double *l_out) {
    const double *qi = q + i * (long)d;
    double m = -INFINITY;
    for (long j = 0; j < Nk; ++j) {
        if (!visible(mk, i, j)) continue;
        double s = score(qi, k + j * (long)d, d, scale);
        if (s > m) m = s;
    }
    double l = 0.0;
    for (long j = 0; j < Nk; ++j) {
        if (!visible(mk, i, j)) continue;
        l += exp(score(qi, k + j * (long)d, d, scale) - m);
    }
    *m_out = m;
    *l_out = l;
}

static Mask make_mask(int causal, int Nq, int Nk, const unsigned char *bm, int bq, int bk) {
    Mask mk = {causal, (long)Nk - Nq, bm, bq, bk, bm ? (Nk + bk - 1) / bk : 0};
    return mk;
}

/*
 * Forward: o = softmax(scale Q K^T [masked]) V and lse, per query head.
 * q, o: [BH][Nq][d]; k, v: [BH/G][Nk][d]; lse: [BH][Nq].  G = group >= 1.
 * bm: block mask [ceil(Nq/bq)][ceil(Nk/bk)] or NULL.
 */
void oracle_attn_fwd(const double *q, const double *k, const double *v,
                     double *o, double *lse, int BH, int Nq, int Nk, int d,
                     double scale, int causal, int group,
                     const unsigned char *bm, int bq, int bk) {
    const long hq = (long)Nq * d, hk = (long)Nk * d;
    const Mask mkv = make_mask(causal, Nq, Nk, bm, bq, bk), *mk = &mkv;
#pragma omp parallel for collapse(2) schedule(dynamic, 4)
    for (int h = 0; h < BH; ++h) {
        for (int i = 0; i < Nq; ++i) {
            const double *qh = q + h * hq, *kh = k + (h / group) * hk, *vh = v + (h / group) * hk;
            double m, l;
            row_stats(qh, kh, i, Nk, mk, d, scale, &m, &l);
            double *oi = o + h * hq + (long)i * d;
            for (int c = 0; c < d; ++c) oi[c] = 0.0;
            for (long j = 0; j < Nk; ++j) {
                if (!visible(mk, i, j)) continue;
                double p = exp(score(qh + (long)i * d, kh + j * d, d, scale) - m) / l;
                const double *vj = vh + j * d;
                for (int c = 0; c < d; ++c) oi[c] += p * vj[c];
            }
            lse[(long)h * Nq + i] = m + log(l);
        }
    }
}

/*
 * Backward: dq, dk, dv of L with dL/dO = dO.
 * q, dO, dq: [BH][Nq][d]; k, v, dk, dv: [BH/G][Nk][d].  Forward quantities
 * are recomputed here from q, k, v (the oracle takes nothing produced by the
 * GPU path).  D_out (may be NULL): [BH][Nq], receives D_i = sum_j p_ij dp_ij.
 * bm: block mask as for the forward, or NULL.
 */
void oracle_attn_bwd(const double *q, const double *k, const double *v,
                     const double *dO, double *dq, double *dk, double *dv,
                     double *D_out, int BH, int Nq, int Nk, int d, double scale,
                     int causal, int group, const unsigned char *bm, int bq, int bk) {
    const long hq = (long)Nq * d, hk = (long)Nk * d;
    const Mask mkv = make_mask(causal, Nq, Nk, bm, bq, bk), *mk = &mkv;
    double *m = (double *)malloc(sizeof(double) * (size_t)BH * Nq);
    double *l = (double *)malloc(sizeof(double) * (size_t)BH * Nq);
    double *D = (double *)malloc(sizeof(double) * (size_t)BH * Nq);

    /* Pass over query rows: row statistics, D_i, and dq_i. */
#pragma omp parallel for collapse(2) schedule(dynamic, 4)
    for (int h = 0; h < BH; ++h) {
        for (int i = 0; i < Nq; ++i) {
            const double *qh = q + h * hq, *kh = k + (h / group) * hk, *vh = v + (h / group) * hk;
            const double *dOi = dO + h * hq + (long)i * d;
            const long r = (long)h * Nq + i;
            row_stats(qh, kh, i, Nk, mk, d, scale, &m[r], &l[r]);
            /* D_i = sum_j p_ij dp_ij */
            double Di = 0.0;
            for (long j = 0; j < Nk; ++j) {
                if (!visible(mk, i, j)) continue;
                double p = exp(score(qh + (long)i * d, kh + j * d, d, scale) - m[r]) / l[r];
                double dp = 0.0;
                for (int c = 0; c < d; ++c) dp += dOi[c] * vh[j * d + c];
                Di += p * dp;
            }
            D[r] = Di;
            /* dq_i = scale * sum_j ds_ij k_j */
            double *dqi = dq + h * hq + (long)i * d;
            for (int c = 0; c < d; ++c) dqi[c] = 0.0;
            for (long j = 0; j < Nk; ++j) {
                if (!visible(mk, i, j)) continue;
                double p = exp(score(qh + (long)i * d, kh + j * d, d, scale) - m[r]) / l[r];
                double dp = 0.0;
                for (int c = 0; c < d; ++c) dp += dOi[c] * vh[j * d + c];
                double ds = p * (dp - Di);
                for (int c = 0; c < d; ++c) dqi[c] += scale * ds * kh[j * d + c];
            }
        }
    }

    /* Pass over keys of each key/value head hk:
     * dv_j = sum over its query heads h and rows i of p_ij dO_i,
     * dk_j = scale * sum over the same of ds_ij q_i. */
    const int BHkv = BH / group;
#pragma omp parallel for collapse(2) schedule(dynamic, 4)
    for (int kv = 0; kv < BHkv; ++kv) {
        for (int j = 0; j < Nk; ++j) {
            const double *kh = k + kv * hk, *vh = v + kv * hk;
            double *dvj = dv + kv * hk + (long)j * d;
            double *dkj = dk + kv * hk + (long)j * d;
            for (int c = 0; c < d; ++c) { dvj[c] = 0.0; dkj[c] = 0.0; }
            for (int g = 0; g < group; ++g) {
                const int h = kv * group + g;
                const double *qh = q + h * hq, *dOh = dO + h * hq;
                for (long i = 0; i < Nq; ++i) {
                    if (!visible(mk, i, j)) continue;
                    const long r = (long)h * Nq + i;
                    double p = exp(score(qh + i * d, kh + (long)j * d, d, scale) - m[r]) / l[r];
                    double dp = 0.0;
                    for (int c = 0; c < d; ++c) dp += dOh[i * d + c] * vh[(long)j * d + c];
                    double ds = p * (dp - D[r]);
                    for (int c = 0; c < d; ++c) {
                        dvj[c] += p * dOh[i * d + c];
                        dkj[c] += scale * ds * qh[i * d + c];
                    }
                }
            }
        }
    }

    if (D_out) {
        for (long r = 0; r < (long)BH * Nq; ++r) D_out[r] = D[r];
    }
    free(m);
    free(l);
    free(D);
}

/*
 * Forward for a chosen subset of query rows of one head (for sampled checks
 * at sizes where the full oracle would take too long).  rows: [R] indices.
 * q: [Nq][d], k, v: [Nk][d] of that head; o: [R][d]; lse: [R].
 */
void oracle_attn_fwd_rows(const double *q, const double *k, const double *v,
                          const int *rows, int R, double *o, double *lse,
                          int Nq, int Nk, int d, double scale, int causal) {
    const Mask mkv = make_mask(causal, Nq, Nk, NULL, 1, 1), *mk = &mkv;
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < R; ++t) {
        const long i = rows[t];
        double m, l;
        row_stats(q, k, i, Nk, mk, d, scale, &m, &l);
        double *oi = o + (long)t * d;
        for (int c = 0; c < d; ++c) oi[c] = 0.0;
        for (long j = 0; j < Nk; ++j) {
            if (!visible(mk, i, j)) continue;
            double p = exp(score(q + i * d, k + j * d, d, scale) - m) / l;
            for (int c = 0; c < d; ++c) oi[c] += p * v[j * d + c];
        }
        lse[t] = m + log(l);
    }
}

/*
 * Backward for chosen rows of one head (for checks at sizes where the full
 * backward would take too long): dq of the query rows qrows[0 .. Rq) and dk,
 * dv of the key rows krows[0 .. Rk), with the formulas of oracle_attn_bwd
 * restricted to those outputs.  One head, no grouping, no block mask; causal
 * with Nq != Nk aligns the last query with the last key as above.
 * q, dO: [Nq][d]; k, v: [Nk][d]; dq: [Rq][d]; dk, dv: [Rk][d].
 *
 * dk_j and dv_j sum over every query row i that sees key j, so the row
 * statistics m_i, l_i and D_i are computed for each such row (and for the
 * rows of qrows); no statistic is taken from elsewhere.
 */
void oracle_attn_bwd_rows(const double *q, const double *k, const double *v, const double *dO,
                          const int *qrows, int Rq, const int *krows, int Rk,
                          double *dq, double *dk, double *dv,
                          int Nq, int Nk, int d, double scale, int causal) {
    const Mask mkv = make_mask(causal, Nq, Nk, NULL, 1, 1), *mk = &mkv;
    double *m = (double *)malloc(sizeof(double) * (size_t)(Nq > 0 ? Nq : 1));
    double *l = (double *)malloc(sizeof(double) * (size_t)(Nq > 0 ? Nq : 1));
    double *D = (double *)malloc(sizeof(double) * (size_t)(Nq > 0 ? Nq : 1));
    unsigned char *need = (unsigned char *)calloc((size_t)(Nq > 0 ? Nq : 1), 1);
    /* a statistic that is used without having been computed shows as NaN */
    for (int i = 0; i < Nq; ++i) m[i] = l[i] = D[i] = NAN;

    /* rows whose statistics are used: the rows of qrows, and every row that
     * sees at least one key of krows */
    for (int t = 0; t < Rq; ++t) need[qrows[t]] = 1;
#pragma omp parallel for schedule(static)
    for (int i = 0; i < Nq; ++i) {
        for (int t = 0; t < Rk && !need[i]; ++t)
            if (visible(mk, i, krows[t])) need[i] = 1;
    }

    /* m_i, l_i (safe softmax) and D_i = sum_j p_ij dp_ij of those rows */
#pragma omp parallel for schedule(dynamic, 4)
    for (int i = 0; i < Nq; ++i) {
        if (!need[i]) continue;
        const double *dOi = dO + (long)i * d;
        row_stats(q, k, i, Nk, mk, d, scale, &m[i], &l[i]);
        double Di = 0.0;
        for (long j = 0; j < Nk; ++j) {
            if (!visible(mk, i, j)) continue;
            double p = exp(score(q + (long)i * d, k + j * d, d, scale) - m[i]) / l[i];
            double dp = 0.0;
            for (int c = 0; c < d; ++c) dp += dOi[c] * v[j * d + c];
            Di += p * dp;
        }
        D[i] = Di;
    }

    /* dq_i = scale * sum_j ds_ij k_j for the rows of qrows */
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < Rq; ++t) {
        const long i = qrows[t];
        const double *dOi = dO + i * d;
        double *dqi = dq + (long)t * d;
        for (int c = 0; c < d; ++c) dqi[c] = 0.0;
        for (long j = 0; j < Nk; ++j) {
            if (!visible(mk, i, j)) continue;
            double p = exp(score(q + i * d, k + j * d, d, scale) - m[i]) / l[i];
            double dp = 0.0;
            for (int c = 0; c < d; ++c) dp += dOi[c] * v[j * d + c];
            double ds = p * (dp - D[i]);
            for (int c = 0; c < d; ++c) dqi[c] += scale * ds * k[j * d + c];
        }
    }

    /* dv_j = sum_i p_ij dO_i and dk_j = scale * sum_i ds_ij q_i for the keys of krows */
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < Rk; ++t) {
        const long j = krows[t];
        double *dvj = dv + (long)t * d, *dkj = dk + (long)t * d;
        for (int c = 0; c < d; ++c) { dvj[c] = 0.0; dkj[c] = 0.0; }
        for (long i = 0; i < Nq; ++i) {
            if (!visible(mk, i, j)) continue;
            double p = exp(score(q + i * d, k + j * d, d, scale) - m[i]) / l[i];
            double dp = 0.0;
            for (int c = 0; c < d; ++c) dp += dO[i * d + c] * v[j * d + c];
            double ds = p * (dp - D[i]);
            for (int c = 0; c < d; ++c) {
                dvj[c] += p * dO[i * d + c];
                dkj[c] += scale * ds * q[i * d + c];
            }
        }
    }
    free(m);
    free(l);
    free(D);
    free(need);
}
