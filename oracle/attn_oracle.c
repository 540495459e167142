/*
 * attn_oracle.c -- fp64 CPU oracle for the multi-head scaled dot-product
 * attention forward pass.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark load this library. The CUDA path never calls it and shares
 * no code, header, constant or helper with it.
 *
 * What it computes is the plain definition, step by step, for every head
 * independently and for every query row i (no tiling, no online rescaling):
 *
 *   s_j   = scale * sum_t q_it k_jt                 scores of row i
 *           ("Transformer 详解" §4.1 steps 2-3; "从 RNN 到 Transformer（二）"
 *            §4.3 steps 2-3 and §4.9: scores = Q Kᵀ / sqrt(d_k))
 *   J     = keys visible to row i under the mask:
 *           none         every j                     (encoder self-attention,
 *                                                     "Transformer 详解" §4.1;
 *                                                     cross-attention §5.4)
 *           causal       j <= i + (m - n)            ("Transformer 详解" §5.3
 *                                                     Mask_ij = 0 if j<=i else
 *                                                     -inf; "第2章：完整的
 *                                                     Transformer 架构" §6; the
 *                                                     pages give the square
 *                                                     case n = m; for n != m
 *                                                     the queries are the last
 *                                                     n positions of the m keys)
 *           key padding  j < len_b, all query rows   ("Transformer 详解" §3.4:
 *                                                     mask [batch,1,1,seq]
 *                                                     broadcasts over heads and
 *                                                     queries, masks keys)
 *           causal and   both conditions             ("Transformer 详解" §5.3:
 *           key padding                               tgt_mask = pad_mask &
 *                                                     subsequent_mask)
 *           causal in    j < len_b and               (a cache of fixed size m
 *           the cache    j <= i + (len_b - n)         filled to len_b positions,
 *                                                     the n queries being its
 *                                                     last n: the wiki page's KV
 *                                                     cache, "实现要点")
 *   mu    = max_{j in J} s_j;  Z = sum_{j in J} exp(s_j - mu)
 *   w_j   = exp(s_j - mu) / Z for j in J, 0 otherwise      (row softmax; the
 *           shift by mu leaves the value unchanged and keeps exp in range)
 *   o_i   = sum_j w_j v_j                            ("从 RNN 到 Transformer（二）"
 *                                                     §4.3 step 5, weighted sum)
 *   LSE_i = mu + ln Z  (natural log of the masked sum of exp of scaled scores)
 *
 * A masked position is excluded from J, which is the -inf fill of the pages'
 * minimal implementation. With at least one visible key the -1e9 fill of
 * "Transformer 详解" §3.4 gives the same result in fp64. A row with no
 * visible key (key length 0) gets o_i = 0 and LSE_i = -inf.
 *
 * Key lengths are clamped to [0, m].
 *
 * Layouts: Q [B,H,n,dk], K [B,H,m,dk], V [B,H,m,dv], O [B,H,n,dv], LSE
 * [B,H,n], all contiguous row-major fp64; key_lengths int32 [B].
 *
 * Backward (oracle_attn_bwd). For a loss whose gradient with respect to O is
 * dO, the chain rule through the definition above gives, per head and row i
 * with at least one visible key (w_j the weights of row i, 0 when masked):
 *
 *   dV_j  += w_j dO_i                                  (o_i = sum_j w_j v_j)
 *   dP_j   = dO_i . v_j
 *   dS_j   = w_j (dP_j - D_i),  D_i = sum_j w_j dP_j   (softmax Jacobian:
 *            dw_j/ds_k = w_j (delta_jk - w_k); D_i also equals dO_i . o_i)
 *   dQ_i   = scale sum_j dS_j k_j,  dK_j += scale dS_j q_i   (s_j = scale q_i.k_j)
 *
 * Rows with no visible key contribute nothing (their o_i = 0 is constant).
 * Masked keys get dK_j = dV_j = 0.
 *
 * Linear distance bias (oracle_attn_fwd_alibi, oracle_attn_rows_alibi).
 * "第2章：完整的 Transformer 架构" §5.3 (ALiBi) subtracts from every scaled
 * score a bias proportional to the distance between query and key, with a
 * slope m_h of its own for each head:
 *
 *   s_j   = scale * q_i . k_j - m_h |i' - j|,   i' = i + (m - n)
 *
 * where i' is the query's position among the keys (the n queries are the last
 * n of the m positions, as for the causal mask; i' = i when n = m). The masks,
 * the softmax, the weighted sum and the LSE then proceed as above on these
 * biased scores. The backward (oracle_attn_bwd_alibi) is the chain rule above
 * with the weights of these biased scores: the bias depends on neither Q nor K,
 * so the formulas for dS, dQ, dK and dV are unchanged.
 *
 * ORACLE_PLANT (compile-time, default 0, 1..11, 14..18) plants one known mistake so
 * that the test suite can show that its pins catch it; the shipped build never
 * sets it.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_PLANT
#define ORACLE_PLANT 0
#endif

enum {
    ORACLE_MASK_NONE = 0,
    ORACLE_MASK_CAUSAL = 1,
    ORACLE_MASK_KEY_PADDING = 2,
    ORACLE_MASK_CAUSAL_KEY_PADDING = 3,
    ORACLE_MASK_CAUSAL_CACHE = 4
};

static int causal_visible(int64_t i, int64_t j, int64_t off)
{
#if ORACLE_PLANT == 2
    return j < i + off;            /* planted: diagonal excluded */
#elif ORACLE_PLANT == 7
    (void)off;
    return j <= i;                 /* planted: diagonal not shifted for n != m */
#else
    return j <= i + off;
#endif
}

static int padding_visible(int64_t i, int64_t j, int64_t len)
{
#if ORACLE_PLANT == 5
    (void)j;
    return i < len;                /* planted: padding applied to queries */
#else
    (void)i;
    return j < len;
#endif
}

/* Is key j visible to query row i? off = m - n aligns the causal diagonal so
 * that the last query row sees every key. */
static int visible(int mask_kind, int64_t i, int64_t j, int64_t len, int64_t off)
{
    switch (mask_kind) {
    case ORACLE_MASK_CAUSAL: return causal_visible(i, j, off);
    case ORACLE_MASK_KEY_PADDING: return padding_visible(i, j, len);
    case ORACLE_MASK_CAUSAL_CACHE: return causal_visible(i, j, off) && padding_visible(i, j, len);
    case ORACLE_MASK_CAUSAL_KEY_PADDING:
#if ORACLE_PLANT == 8
        return causal_visible(i, j, off) || padding_visible(i, j, len);  /* planted: union */
#else
        return causal_visible(i, j, off) && padding_visible(i, j, len);
#endif
    default: return 1;
    }
}

static int uses_lengths(int mask_kind)
{
    return mask_kind == ORACLE_MASK_KEY_PADDING || mask_kind == ORACLE_MASK_CAUSAL_KEY_PADDING ||
           mask_kind == ORACLE_MASK_CAUSAL_CACHE;
}

/* Offset of row i's position among the keys: the n queries are the last n of the m
 * keys, or of the first len keys under the cache mask (position i + off). */
static int64_t row_offset(int mask_kind, int64_t m, int64_t n, int64_t len)
{
#if ORACLE_PLANT == 18
    (void)mask_kind;
    (void)len;
    return m - n;                  /* planted: cache mask aligned to m, not to the length */
#else
    return mask_kind == ORACLE_MASK_CAUSAL_CACHE ? len - n : m - n;
#endif
}

static int64_t clamp_len(const int32_t* key_lengths, int mask_kind, int64_t b, int64_t m)
{
    if (!uses_lengths(mask_kind) || key_lengths == NULL) return m;
    int64_t len = key_lengths[b];
    if (len < 0) len = 0;
    if (len > m) len = m;
    return len;
}

/*
 * One query row of one head. q [dk], Kh [m,dk], Vh [m,dv] belong to that head.
 * s and w are caller scratch of m doubles. Writes o [dv], *lse, and, if w_out
 * is not NULL, the m attention weights of the row.
 */
static void attn_row(const double* q, const double* Kh, const double* Vh, int64_t m,
                     int dk, int dv, int mask_kind, int64_t i, int64_t len, int64_t off,
                     double scale, double slope, double* s, double* o, double* lse, double* w_out)
{
    /* 1. scaled scores of every key */
    for (int64_t j = 0; j < m; ++j) {
        double dot = 0.0;
        for (int t = 0; t < dk; ++t) {
#if ORACLE_PLANT == 3
            dot += q[t] * Kh[(int64_t)t * dk + (j % dk)];   /* planted: wrong K index */
#else
            dot += q[t] * Kh[j * dk + t];
#endif
        }
#if ORACLE_PLANT == 1
        s[j] = dot;                /* planted: scale dropped */
#else
        s[j] = scale * dot;
#endif
        /* linear distance bias (zero slope: none) */
#if ORACLE_PLANT == 14
        s[j] += slope * fabs((double)(i + off - j));    /* planted: bias added */
#elif ORACLE_PLANT == 15
        s[j] -= slope * fabs((double)(i - j));          /* planted: query position not aligned */
#else
        s[j] -= slope * fabs((double)(i + off - j));
#endif
    }
    /* 2. maximum over the visible keys */
    double mu = -INFINITY;
    int64_t count = 0;
    for (int64_t j = 0; j < m; ++j) {
        if (!visible(mask_kind, i, j, len, off)) continue;
        if (s[j] > mu) mu = s[j];
        ++count;
    }
    for (int c = 0; c < dv; ++c) o[c] = 0.0;
    if (count == 0) {
        *lse = -INFINITY;
        if (w_out) for (int64_t j = 0; j < m; ++j) w_out[j] = 0.0;
        return;
    }
    /* 3. normaliser and weights */
    double Z = 0.0;
    for (int64_t j = 0; j < m; ++j)
        if (visible(mask_kind, i, j, len, off)) Z += exp(s[j] - mu);
    for (int64_t j = 0; j < m; ++j) {
        double wj = visible(mask_kind, i, j, len, off) ? exp(s[j] - mu) / Z : 0.0;
#if ORACLE_PLANT == 6
        if (j == 0) wj = 0.0;      /* planted: first key dropped from the sum */
#endif
        s[j] = wj;
        if (w_out) w_out[j] = wj;
    }
    /* 4. weighted sum of the values, and the logsumexp */
    for (int64_t j = 0; j < m; ++j) {
        if (s[j] == 0.0) continue;
        const double* v = Vh + j * dv;
        for (int c = 0; c < dv; ++c) o[c] += s[j] * v[c];
    }
#if ORACLE_PLANT == 4
    *lse = log(Z);                 /* planted: max shift not added back */
#else
    *lse = mu + log(Z);
#endif
}

typedef struct {
    const double *Q, *K, *V;
    const int32_t* key_lengths;
    int64_t B, H, n, m;
    int dk, dv, mask_kind;
    double scale;
    const double* slopes;  /* per head [H], or NULL: no distance bias */
    double *O, *LSE, *W;
    const int64_t* rows;   /* NULL: all rows; else flat indices into [B*H*n] */
    int64_t nrows;
    int nthreads, tid;
} job_t;

/* Distance-bias slope of head h of batch entry b (0 without a bias). */
static double head_slope(const job_t* jb, int64_t b, int64_t h)
{
    if (jb->slopes == NULL) return 0.0;
#if ORACLE_PLANT == 16
    (void)h;
    return jb->slopes[b % jb->H];                 /* planted: slope indexed by batch entry */
#else
    (void)b;
    return jb->slopes[h];
#endif
}

static void* worker(void* arg)
{
    job_t* jb = (job_t*)arg;
    double* s = (double*)malloc(sizeof(double) * (size_t)(jb->m > 0 ? jb->m : 1));
    if (!s) return (void*)1;
    if (jb->rows == NULL) {
        /* every (b,h) pair this thread owns, every row of it */
        for (int64_t bh = jb->tid; bh < jb->B * jb->H; bh += jb->nthreads) {
            int64_t b = bh / jb->H;
            int64_t len = clamp_len(jb->key_lengths, jb->mask_kind, b, jb->m);
            double slope = head_slope(jb, b, bh % jb->H);
            const double* Kh = jb->K + bh * jb->m * jb->dk;
            const double* Vh = jb->V + bh * jb->m * jb->dv;
            for (int64_t i = 0; i < jb->n; ++i) {
                int64_t r = bh * jb->n + i;
                attn_row(jb->Q + r * jb->dk, Kh, Vh, jb->m, jb->dk, jb->dv, jb->mask_kind, i,
                         len, row_offset(jb->mask_kind, jb->m, jb->n, len), jb->scale, slope, s,
                         jb->O + r * jb->dv, jb->LSE + r,
                         jb->W ? jb->W + r * jb->m : NULL);
            }
        }
    } else {
        /* sampled rows: output k of O/LSE belongs to flat row rows[k] */
        for (int64_t k = jb->tid; k < jb->nrows; k += jb->nthreads) {
            int64_t r = jb->rows[k];
            int64_t bh = r / jb->n, i = r % jb->n, b = bh / jb->H;
            int64_t len = clamp_len(jb->key_lengths, jb->mask_kind, b, jb->m);
            attn_row(jb->Q + r * jb->dk, jb->K + bh * jb->m * jb->dk,
                     jb->V + bh * jb->m * jb->dv, jb->m, jb->dk, jb->dv, jb->mask_kind, i, len,
                     row_offset(jb->mask_kind, jb->m, jb->n, len), jb->scale, head_slope(jb, b, bh % jb->H), s,
                     jb->O + k * jb->dv, jb->LSE + k, NULL);
        }
    }
    free(s);
    return NULL;
}

static int run(job_t base)
{
    int nt = base.nthreads < 1 ? 1 : base.nthreads;
    if (nt > 1024) nt = 1024;
    pthread_t th[1024];
    job_t jobs[1024];
    int rc = 0;
    for (int t = 0; t < nt; ++t) {
        jobs[t] = base;
        jobs[t].nthreads = nt;
        jobs[t].tid = t;
    }
    if (nt == 1) return worker(&jobs[0]) == NULL ? 0 : -1;
    int started = 0;
    for (int t = 0; t < nt; ++t) {
        if (pthread_create(&th[t], NULL, worker, &jobs[t]) != 0) { rc = -1; break; }
        ++started;
    }
    for (int t = 0; t < started; ++t) {
        void* ret = NULL;
        pthread_join(th[t], &ret);
        if (ret != NULL) rc = -1;
    }
    return rc;
}

/*
 * Backward of one head. Qh [n,dk], Kh [m,dk], Vh [m,dv], dOh [n,dv]; writes
 * dQh [n,dk], dKh [m,dk], dVh [m,dv]. w, dp are scratch of m doubles, o of dv.
 */
static void head_bwd(const double* Qh, const double* Kh, const double* Vh, const double* dOh,
                     int64_t n, int64_t m, int dk, int dv, int mask_kind, int64_t len, double scale,
                     double slope, double* dQh, double* dKh, double* dVh, double* w, double* dp, double* o)
{
#if ORACLE_PLANT == 17
    slope = 0.0;                   /* planted: distance bias dropped in the backward */
#endif
    for (int64_t t = 0; t < m * dk; ++t) dKh[t] = 0.0;
    for (int64_t t = 0; t < m * dv; ++t) dVh[t] = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        const double* q = Qh + i * dk;
        const double* g = dOh + i * dv;
        double* dq = dQh + i * dk;
        double lse;
        for (int c = 0; c < dk; ++c) dq[c] = 0.0;
        /* forward of row i: on return w holds its weights (0 where masked) */
        attn_row(q, Kh, Vh, m, dk, dv, mask_kind, i, len, row_offset(mask_kind, m, n, len), scale, slope, w, o,
                 &lse, NULL);
        if (isinf(lse)) continue;          /* no visible key: o_i = 0 is constant */
        double D = 0.0;
        for (int64_t j = 0; j < m; ++j) {
            double acc = 0.0;
            const double* v = Vh + j * dv;
            for (int c = 0; c < dv; ++c) acc += g[c] * v[c];
            dp[j] = acc;
            D += w[j] * acc;
        }
        for (int64_t j = 0; j < m; ++j) {
            if (w[j] == 0.0) continue;
#if ORACLE_PLANT == 9
            double ds = w[j] * dp[j];                      /* planted: D_i dropped */
#else
            double ds = w[j] * (dp[j] - D);
#endif
            const double* k = Kh + j * dk;
            double* dk_j = dKh + j * dk;
            double* dv_j = dVh + j * dv;
            for (int c = 0; c < dk; ++c) {
                dq[c] += scale * ds * k[c];
#if ORACLE_PLANT == 10
                dk_j[c] += ds * q[c];                      /* planted: scale dropped in dK */
#else
                dk_j[c] += scale * ds * q[c];
#endif
            }
#if ORACLE_PLANT == 11
            for (int c = 0; c < dv; ++c) dv_j[c] += w[j] * o[c];  /* planted: O in place of dO */
#else
            for (int c = 0; c < dv; ++c) dv_j[c] += w[j] * g[c];
#endif
        }
    }
}

typedef struct {
    const double *Q, *K, *V, *dO;
    const int32_t* key_lengths;
    int64_t B, H, n, m;
    int dk, dv, mask_kind;
    double scale;
    const double* slopes;  /* per head [H], or NULL: no distance bias */
    double *dQ, *dK, *dV;
    int nthreads, tid;
} bwd_job_t;

static void* bwd_worker(void* arg)
{
    bwd_job_t* jb = (bwd_job_t*)arg;
    size_t mm = (size_t)(jb->m > 0 ? jb->m : 1);
    double* w = (double*)malloc(sizeof(double) * mm);
    double* dp = (double*)malloc(sizeof(double) * mm);
    double* o = (double*)malloc(sizeof(double) * (size_t)jb->dv);
    void* ret = NULL;
    if (!w || !dp || !o) {
        ret = (void*)1;
    } else {
        for (int64_t bh = jb->tid; bh < jb->B * jb->H; bh += jb->nthreads) {
            int64_t len = clamp_len(jb->key_lengths, jb->mask_kind, bh / jb->H, jb->m);
            head_bwd(jb->Q + bh * jb->n * jb->dk, jb->K + bh * jb->m * jb->dk,
                     jb->V + bh * jb->m * jb->dv, jb->dO + bh * jb->n * jb->dv, jb->n, jb->m,
                     jb->dk, jb->dv, jb->mask_kind, len, jb->scale,
                     jb->slopes ? jb->slopes[bh % jb->H] : 0.0, jb->dQ + bh * jb->n * jb->dk,
                     jb->dK + bh * jb->m * jb->dk, jb->dV + bh * jb->m * jb->dv, w, dp, o);
        }
    }
    free(w);
    free(dp);
    free(o);
    return ret;
}

static int bad_args(int64_t B, int64_t H, int64_t n, int64_t m, int dk, int dv, int mask_kind)
{
    return B < 0 || H < 0 || n < 0 || m < 0 || dk < 1 || dv < 1 || mask_kind < 0 ||
           mask_kind > 4;
}

/* Full forward: O [B,H,n,dv] and LSE [B,H,n]. W (optional, [B,H,n,m]) gets the
 * attention weights for small debugging cases. Returns 0 on success. */
int oracle_attn_fwd(const double* Q, const double* K, const double* V, int64_t B, int64_t H,
                    int64_t n, int64_t m, int dk, int dv, int mask_kind,
                    const int32_t* key_lengths, double scale, double* O, double* LSE,
                    double* W, int nthreads)
{
    if (bad_args(B, H, n, m, dk, dv, mask_kind)) return -1;
    if (uses_lengths(mask_kind) && key_lengths == NULL) return -1;
    job_t jb = {Q, K, V, key_lengths, B, H, n, m, dk, dv, mask_kind, scale, NULL, O, LSE, W,
                NULL, 0, nthreads, 0};
    return run(jb);
}

/* Forward with the linear distance bias: slopes [H] holds m_h of every head. */
int oracle_attn_fwd_alibi(const double* Q, const double* K, const double* V, int64_t B,
                          int64_t H, int64_t n, int64_t m, int dk, int dv, int mask_kind,
                          const int32_t* key_lengths, const double* slopes, double scale,
                          double* O, double* LSE, double* W, int nthreads)
{
    if (bad_args(B, H, n, m, dk, dv, mask_kind) || slopes == NULL) return -1;
    if (uses_lengths(mask_kind) && key_lengths == NULL) return -1;
    job_t jb = {Q, K, V, key_lengths, B, H, n, m, dk, dv, mask_kind, scale, slopes, O, LSE, W,
                NULL, 0, nthreads, 0};
    return run(jb);
}

/* Selected rows only: rows[k] is a flat index b*H*n + h*n + i; O is [nrows,dv]
 * and LSE [nrows]. Used to check full-size outputs one row at a time. */
int oracle_attn_rows(const double* Q, const double* K, const double* V, int64_t B, int64_t H,
                     int64_t n, int64_t m, int dk, int dv, int mask_kind,
                     const int32_t* key_lengths, double scale, const int64_t* rows,
                     int64_t nrows, double* O, double* LSE, int nthreads)
{
    if (bad_args(B, H, n, m, dk, dv, mask_kind) || rows == NULL || nrows < 0) return -1;
    if (uses_lengths(mask_kind) && key_lengths == NULL) return -1;
    for (int64_t k = 0; k < nrows; ++k)
        if (rows[k] < 0 || rows[k] >= B * H * n) return -1;
    job_t jb = {Q, K, V, key_lengths, B, H, n, m, dk, dv, mask_kind, scale, NULL, O, LSE, NULL,
                rows, nrows, nthreads, 0};
    return run(jb);
}

/* Selected rows with the linear distance bias (slopes [H]). */
int oracle_attn_rows_alibi(const double* Q, const double* K, const double* V, int64_t B,
                           int64_t H, int64_t n, int64_t m, int dk, int dv, int mask_kind,
                           const int32_t* key_lengths, const double* slopes, double scale,
                           const int64_t* rows, int64_t nrows, double* O, double* LSE,
                           int nthreads)
{
    if (bad_args(B, H, n, m, dk, dv, mask_kind) || rows == NULL || nrows < 0 || slopes == NULL)
        return -1;
    if (uses_lengths(mask_kind) && key_lengths == NULL) return -1;
    for (int64_t k = 0; k < nrows; ++k)
        if (rows[k] < 0 || rows[k] >= B * H * n) return -1;
    job_t jb = {Q, K, V, key_lengths, B, H, n, m, dk, dv, mask_kind, scale, slopes, O, LSE, NULL,
                rows, nrows, nthreads, 0};
    return run(jb);
}

/* Backward of every head; slopes may be NULL (no distance bias). */
static int bwd_impl(const double* Q, const double* K, const double* V, const double* dO, int64_t B,
                    int64_t H, int64_t n, int64_t m, int dk, int dv, int mask_kind,
                    const int32_t* key_lengths, const double* slopes, double scale, double* dQ,
                    double* dK, double* dV, int nthreads)
{
    if (bad_args(B, H, n, m, dk, dv, mask_kind)) return -1;
    if (uses_lengths(mask_kind) && key_lengths == NULL) return -1;
    int nt = nthreads < 1 ? 1 : (nthreads > 1024 ? 1024 : nthreads);
    pthread_t th[1024];
    bwd_job_t jobs[1024];
    int rc = 0, started = 0;
    for (int t = 0; t < nt; ++t) {
        bwd_job_t jb = {Q, K, V, dO, key_lengths, B, H, n, m, dk, dv, mask_kind, scale,
                        slopes, dQ, dK, dV, nt, t};
        jobs[t] = jb;
    }
    if (nt == 1) return bwd_worker(&jobs[0]) == NULL ? 0 : -1;
    for (int t = 0; t < nt; ++t) {
        if (pthread_create(&th[t], NULL, bwd_worker, &jobs[t]) != 0) { rc = -1; break; }
        ++started;
    }
    for (int t = 0; t < started; ++t) {
        void* ret = NULL;
        pthread_join(th[t], &ret);
        if (ret != NULL) rc = -1;
    }
    return rc;
}

/* Backward: dQ [B,H,n,dk], dK [B,H,m,dk], dV [B,H,m,dv] for the upstream
 * gradient dO [B,H,n,dv]. Returns 0 on success. */
int oracle_attn_bwd(const double* Q, const double* K, const double* V, const double* dO,
                    int64_t B, int64_t H, int64_t n, int64_t m, int dk, int dv, int mask_kind,
                    const int32_t* key_lengths, double scale, double* dQ, double* dK, double* dV,
                    int nthreads)
{
    return bwd_impl(Q, K, V, dO, B, H, n, m, dk, dv, mask_kind, key_lengths, NULL, scale, dQ, dK, dV,
                    nthreads);
}

/* Backward of the forward with the linear distance bias (slopes [H]). */
int oracle_attn_bwd_alibi(const double* Q, const double* K, const double* V, const double* dO,
                          int64_t B, int64_t H, int64_t n, int64_t m, int dk, int dv, int mask_kind,
                          const int32_t* key_lengths, const double* slopes, double scale, double* dQ,
                          double* dK, double* dV, int nthreads)
{
    if (slopes == NULL) return -1;
    return bwd_impl(Q, K, V, dO, B, H, n, m, dk, dv, mask_kind, key_lengths, slopes, scale, dQ, dK, dV,
                    nthreads);
}
