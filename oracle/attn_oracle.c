/*
 * attn_oracle.c -- plain, slow, fp64 CPU attention.  TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the CPU-baseline leg of the bench
 * load this file's shared library.  The product path (the CUDA library and its
 * Python binding) never links, imports or calls it, and it shares no code,
 * header, table or constant with that path.
 *
 * What it computes is the textbook definition of scaled-dot-product attention
 * that the pages describe in words:
 *   - flash-attention-cuda README, "What is Attention?": each query weighs every
 *     visible key ("Student 5 pays different amounts of attention to each
 *     previous student"), the weights are percentages that sum to one, and the
 *     answer is the weighted combination of the values;
 *   - same README, "The Problem": the naive method materialises the whole score
 *     table.  The oracle does exactly that (one explicit row of scores at a
 *     time) -- it is the "explicit scores" method, not the tiled one;
 *   - same README, "What did I implement?" (generation phase): a decode query
 *     attends over the first seq_len rows of its KV cache;
 *   - "Kernel design" table, causal row: key j is visible to query i iff j <= i.
 *     When there are fewer queries than keys (a new chunk of a prompt over
 *     keys that already include earlier tokens) the queries are the LAST n_q
 *     positions: key j is visible to query i iff j <= i + (n_k - n_q).  This
 *     is the reading under which a decode row (n_q = 1) sees its whole cache,
 *     as "What did I implement?" describes; for n_q == n_k it is j <= i.
 *
 * For query row i with visible key set J:
 *     s_j  = scale * sum_c Q[i,c] * K[j,c]            (j in J)
 *     m    = max_j s_j
 *     e_j  = exp(s_j - m)
 *     Z    = sum_j e_j
 *     O[i] = sum_j (e_j / Z) * V[j]
 * All arithmetic is IEEE double, accumulated in index order.  Subtracting m
 * does not change the result mathematically; it only keeps exp() in range.
 * An empty visible set gives a zero row (the library's convention for a
 * zero-length cache).  No blocking, no online recurrence, no splitting.
 *
 * Parity pins (tests/test_oracle_pins.py): closed forms on tiny inputs, rows of
 * the weights summing to one, Q=0 giving the mean of the visible values,
 * identical value rows, causal row 0 = V[0], decode(t) = causal prefill row t,
 * shift / permutation / affine invariances, the page's classroom example, and
 * an independent library implementation in float64.
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>

/* Scores of one query row against keys [0, n_vis): s[j] = scale * q . k_j. */
static void score_row(const double *q, const double *k, long n_vis, int d,
                      double scale, double *s) {
    for (long j = 0; j < n_vis; ++j) {
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += q[c] * k[j * (long)d + c];
        s[j] = scale * dot;
    }
}

/* Softmax of s[0..n) in place (max-subtracted); returns 0, or -1 if n == 0. */
static int softmax_inplace(double *s, long n) {
    if (n <= 0) return -1;
    double m = s[0];
    for (long j = 1; j < n; ++j)
        if (s[j] > m) m = s[j];
    double z = 0.0;
    for (long j = 0; j < n; ++j) {
        s[j] = exp(s[j] - m);
        z += s[j];
    }
    for (long j = 0; j < n; ++j) s[j] = s[j] / z;
    return 0;
}

/* out[c] = sum_j p[j] * v[j, c]  over j in [0, n). */
static void weighted_values(const double *p, const double *v, long n, int d,
                            double *out) {
    for (int c = 0; c < d; ++c) out[c] = 0.0;
    for (long j = 0; j < n; ++j)
        for (int c = 0; c < d; ++c) out[c] += p[j] * v[j * (long)d + c];
}

/*
 * One attention head, a chosen subset of query rows.
 *   q: [n_q][d], k, v: [n_k][d], out: [n_rows][d]
 *   rows: the query indices to compute (NULL = all n_q rows, in order)
 *   causal: key j visible to query i iff j <= i + (n_k - n_q)  (j <= i when
 *           n_q == n_k); a row with no visible key is a zero row
 *   p_out: optional [n_rows][n_k] softmax weights (zero for masked keys)
 * Returns 0 on success, -1 on bad arguments or allocation failure.
 */
int oracle_attention_head(const double *q, const double *k, const double *v,
                          double *out, long n_q, long n_k, int d, int causal,
                          double scale, const long *rows, long n_rows,
                          double *p_out) {
    if (d <= 0 || n_q < 0 || n_k < 0) return -1;
    if (rows == NULL) n_rows = n_q;
    double *s = (double *)malloc(sizeof(double) * (size_t)(n_k > 0 ? n_k : 1));
    if (!s) return -1;
    for (long r = 0; r < n_rows; ++r) {
        long i = rows ? rows[r] : r;
        if (i < 0 || i >= n_q) { free(s); return -1; }
        long n_vis = n_k;
        if (causal) {
            n_vis = i + 1 + (n_k - n_q);
            if (n_vis > n_k) n_vis = n_k;
            if (n_vis < 0) n_vis = 0;
        }
        double *o = out + r * (long)d;
        if (p_out)
            for (long j = 0; j < n_k; ++j) p_out[r * n_k + j] = 0.0;
        if (n_vis <= 0) {
            for (int c = 0; c < d; ++c) o[c] = 0.0;
            continue;
        }
        score_row(q + i * (long)d, k, n_vis, d, scale, s);
        softmax_inplace(s, n_vis);
        weighted_values(s, v, n_vis, d, o);
        if (p_out)
            for (long j = 0; j < n_vis; ++j) p_out[r * n_k + j] = s[j];
    }
    free(s);
    return 0;
}

/*
 * Decode for one (batch, head): a single query row q[d] over the first
 * seq_len rows of the cache (k_cache, v_cache: [max_len][d]).  seq_len is
 * clamped to [0, max_len]; seq_len == 0 gives a zero row.
 */
int oracle_decode_head(const double *q, const double *k_cache,
                       const double *v_cache, long seq_len, long max_len, int d,
                       double scale, double *out) {
    if (d <= 0 || max_len < 0) return -1;
    long n = seq_len < 0 ? 0 : (seq_len > max_len ? max_len : seq_len);
    if (n == 0) {
        for (int c = 0; c < d; ++c) out[c] = 0.0;
        return 0;
    }
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    if (!s) return -1;
    score_row(q, k_cache, n, d, scale, s);
    softmax_inplace(s, n);
    weighted_values(s, v_cache, n, d, out);
    free(s);
    return 0;
}

/*
 * Log-sum-exp of every visible score row (the quantity a backward pass needs
 * to recompute the weights): lse_i = log sum_{j visible} exp(s_ij), with
 * s_ij = scale * q_i . k_j and the causal visibility of oracle_attention_head.
 * A row with no visible key gets -INFINITY.
 */
int oracle_lse_head(const double *q, const double *k, long n_q, long n_k, int d, int causal,
                    double scale, double *lse) {
    if (d <= 0 || n_q < 0 || n_k < 0) return -1;
    double *s = (double *)malloc(sizeof(double) * (size_t)(n_k > 0 ? n_k : 1));
    if (!s) return -1;
    for (long i = 0; i < n_q; ++i) {
        long n_vis = n_k;
        if (causal) {
            n_vis = i + 1 + (n_k - n_q);
            if (n_vis > n_k) n_vis = n_k;
            if (n_vis < 0) n_vis = 0;
        }
        if (n_vis == 0) {
            lse[i] = -INFINITY;
            continue;
        }
        score_row(q + i * (long)d, k, n_vis, d, scale, s);
        double m = s[0];
        for (long j = 1; j < n_vis; ++j)
            if (s[j] > m) m = s[j];
        double z = 0.0;
        for (long j = 0; j < n_vis; ++j) z += exp(s[j] - m);
        lse[i] = m + log(z);
    }
    free(s);
    return 0;
}

/*
 * Gradients of one head of O = softmax(scale * Q K^T [mask]) V with respect to
 * Q, K and V, given dO (the backward pass that the flash-attention-cuda README
 * lists under "Future work").  The chain rule through the definition:
 *   P_ij   = softmax weights (as in oracle_attention_head; 0 where masked)
 *   dV_j   = sum_i P_ij dO_i
 *   dP_ij  = dO_i . V_j
 *   dS_ij  = P_ij (dP_ij - sum_k P_ik dP_ik)        (softmax Jacobian)
 *   dQ_i   = scale * sum_j dS_ij K_j
 *   dK_j   = scale * sum_i dS_ij Q_i
 * Explicit n_q x n_k tables, fp64, index order.  Rows with no visible key
 * contribute nothing.
 */
int oracle_backward_head(const double *q, const double *k, const double *v, const double *dout,
                         long n_q, long n_k, int d, int causal, double scale, double *dq, double *dk,
                         double *dv) {
    if (d <= 0 || n_q < 0 || n_k < 0) return -1;
    double *p = (double *)malloc(sizeof(double) * (size_t)(n_k > 0 ? n_k : 1));
    double *dp = (double *)malloc(sizeof(double) * (size_t)(n_k > 0 ? n_k : 1));
    if (!p || !dp) { free(p); free(dp); return -1; }
    for (long x = 0; x < n_q * (long)d; ++x) dq[x] = 0.0;
    for (long x = 0; x < n_k * (long)d; ++x) { dk[x] = 0.0; dv[x] = 0.0; }
    for (long i = 0; i < n_q; ++i) {
        long n_vis = n_k;
        if (causal) {
            n_vis = i + 1 + (n_k - n_q);
            if (n_vis > n_k) n_vis = n_k;
            if (n_vis < 0) n_vis = 0;
        }
        if (n_vis == 0) continue;
        const double *qi = q + i * (long)d, *doi = dout + i * (long)d;
        score_row(qi, k, n_vis, d, scale, p);
        softmax_inplace(p, n_vis);
        double rowdot = 0.0;
        for (long j = 0; j < n_vis; ++j) {
            double t = 0.0;
            for (int c = 0; c < d; ++c) t += doi[c] * v[j * (long)d + c];
            dp[j] = t;
            rowdot += p[j] * t;
        }
        for (long j = 0; j < n_vis; ++j) {
            const double ds = p[j] * (dp[j] - rowdot);
            for (int c = 0; c < d; ++c) {
                dv[j * (long)d + c] += p[j] * doi[c];
                dq[i * (long)d + c] += scale * ds * k[j * (long)d + c];
                dk[j * (long)d + c] += scale * ds * qi[c];
            }
        }
    }
    free(p);
    free(dp);
    return 0;
}
