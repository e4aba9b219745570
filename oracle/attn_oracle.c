/*
 * Test infrastructure -- NOT part of the product path.
 *
 * Plain, slow fp64 CPU statement of masked scaled dot-product attention,
 *
 *     Attention(Q, K, V) = softmax(Q K^T / sqrt(d_k) + M) V,
 *
 * written from "Paper Deep Reading: Attention Is All You Need", §04 Attention
 * mechanics (the attention equation with the additive mask M, and the note
 * that the encoder masks padding while the decoder also masks future
 * positions), and the "Attention Is All You Need" slide deck, "Scaled
 * Dot-Product Attention".  The decoder mask is the one of §03 ("Decoder
 * layer": illegal future connections are set to -inf before the softmax).
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may
 * load this library.  It shares no code, header or constant generator with
 * the CUDA library; the mask flag values below mirror the library's public
 * enum because both describe the same caller-visible argument.
 *
 * Readings of the pages taken here:
 *  - key padding is trailing: key j of batch b is masked iff j >= len_b, the
 *    same for every head; len_b is clamped to [0, n]; query rows are never
 *    masked by padding;
 *  - causal masks key j for query i iff j > i (queries and keys share
 *    positions; the library rejects causal with m != n);
 *  - a query row with no allowed key has output 0 (the formula gives 0/0);
 *  - the scale is an argument (1/sqrt(d_k) in the formula; the pages' worked
 *    example needs other values);
 *  - restricted self-attention (the deep-reading page's §04 complexity table,
 *    "Restricted self-attention", O(r n d); the slide deck's "Limitations and
 *    Future Work") keeps, for query i, the keys j with |i - j| <= w: a
 *    neighbourhood of r = 2w + 1 positions around the query (w is the argument).
 *
 * Every function is the plain definition: no blocking, no online softmax,
 * no reordering beyond what the definition states.  Rows run in parallel with
 * OpenMP when it is available; each row's arithmetic is sequential.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_MASK_KEY_PADDING 1
#define ORACLE_MASK_CAUSAL 2
#define ORACLE_MASK_WINDOW 4

/* bf16 is the upper half of an IEEE binary32: shift the 16 bits into place. */
void oracle_bf16_to_f64(const uint16_t *src, double *dst, int64_t count)
{
    for (int64_t t = 0; t < count; ++t) {
        uint32_t bits = ((uint32_t)src[t]) << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        dst[t] = (double)f;
    }
}

void oracle_f32_to_f64(const float *src, double *dst, int64_t count)
{
    for (int64_t t = 0; t < count; ++t) dst[t] = (double)src[t];
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads the row loops use from now on (for timing the oracle on one core or all). */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Half-width of the restricted-attention window for the current call (set by the
 * _w entry points for the duration of one call; 0 otherwise). */
static int64_t g_window = 0;

/* M_ij == 0 (allowed) or -inf (masked): deep reading §04, §03 "Decoder layer". */
static int key_allowed(int mask_kind, int64_t i, int64_t j, int64_t len_b)
{
    if ((mask_kind & ORACLE_MASK_CAUSAL) && j > i) return 0;
    if ((mask_kind & ORACLE_MASK_KEY_PADDING) && j >= len_b) return 0;
    if ((mask_kind & ORACLE_MASK_WINDOW) && (i - j > g_window || j - i > g_window)) return 0;
    return 1;
}

/*
 * One output row o[0..d) for query row q[0..d) at position i against the
 * keys/values of its (batch, head): Kh, Vh are [n][d].  w is scratch [n].
 */
static void attention_row(const double *q, const double *Kh, const double *Vh,
                          int64_t n, int64_t d, int64_t i, int mask_kind,
                          int64_t len_b, double scale, double *o, double *w)
{
    /* 1. scaled scores s_j = scale * (q . k_j) for every allowed key j */
    int any = 0;
    double mu = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        if (!key_allowed(mask_kind, i, j, len_b)) continue;
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c) dot += q[c] * Kh[j * d + c];
        w[j] = scale * dot;
        if (w[j] > mu) mu = w[j];
        any = 1;
    }
    for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
    if (!any) return; /* fully masked row: 0 */

    /* 2. softmax over the allowed keys: exp(s_j - max) / sum */
    double Z = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        if (!key_allowed(mask_kind, i, j, len_b)) continue;
        w[j] = exp(w[j] - mu);
        Z += w[j];
    }

    /* 3. weighted sum of the value rows */
    for (int64_t j = 0; j < n; ++j) {
        if (!key_allowed(mask_kind, i, j, len_b)) continue;
        double p = w[j] / Z;
        for (int64_t c = 0; c < d; ++c) o[c] += p * Vh[j * d + c];
    }
}

static int64_t clamp_len(const int32_t *key_lengths, int mask_kind, int64_t b, int64_t n)
{
    if (!(mask_kind & ORACLE_MASK_KEY_PADDING) || key_lengths == NULL) return n;
    int64_t len = key_lengths[b];
    if (len < 0) len = 0;
    if (len > n) len = n;
    return len;
}

/*
 * Rows selected by linear id r = ((b*h + head)*m + i), written to out[t][d]
 * for the t-th id.  Q is [B][h][m][d], K and V are [B][h][n][d].
 * Returns 0 on success, -1 on bad arguments or allocation failure.
 */
int oracle_attn_rows(const double *Q, const double *K, const double *V,
                     const int32_t *key_lengths, int mask_kind, double scale,
                     int64_t B, int64_t h, int64_t m, int64_t n, int64_t d,
                     const int64_t *rows, int64_t nrows, double *out)
{
    if (!Q || !K || !V || !out || !rows || B < 0 || h < 0 || m < 0 || n < 1 || d < 1) return -1;
    int failed = 0;
#ifdef _OPENMP
#pragma omp parallel
#endif
    {
        double *w = (double *)malloc(sizeof(double) * (size_t)n);
        if (!w) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
            for (int64_t t = 0; t < nrows; ++t) {
                int64_t r = rows[t];
                int64_t i = r % m;
                int64_t bh = r / m;
                int64_t b = bh / h;
                const double *q = Q + r * d;
                const double *Kh = K + bh * n * d;
                const double *Vh = V + bh * n * d;
                attention_row(q, Kh, Vh, n, d, i, mask_kind,
                              clamp_len(key_lengths, mask_kind, b, n), scale,
                              out + t * d, w);
            }
            free(w);
        }
    }
    return failed ? -1 : 0;
}

/* Every row: out is [B][h][m][d]. */
int oracle_attn_fwd(const double *Q, const double *K, const double *V,
                    const int32_t *key_lengths, int mask_kind, double scale,
                    int64_t B, int64_t h, int64_t m, int64_t n, int64_t d,
                    double *out)
{
    int64_t total = B * h * m;
    int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)(total > 0 ? total : 1));
    if (!rows) return -1;
    for (int64_t r = 0; r < total; ++r) rows[r] = r;
    int rc = oracle_attn_rows(Q, K, V, key_lengths, mask_kind, scale, B, h, m, n, d,
                              rows, total, out);
    free(rows);
    return rc;
}

/*
 * Natural log of the softmax normaliser of every row, lse_i = log sum_j exp(s_ij)
 * over the allowed keys (s_ij the scaled scores above), so that the weights are
 * exp(s_ij - lse_i); -inf for a row with no allowed key.  lse is [B][h][m].
 */
int oracle_attn_lse(const double *Q, const double *K, const int32_t *key_lengths, int mask_kind,
                    double scale, int64_t B, int64_t h, int64_t m, int64_t n, int64_t d, double *lse)
{
    if (!Q || !K || !lse || B < 0 || h < 0 || m < 0 || n < 1 || d < 1) return -1;
    int64_t total = B * h * m;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 16)
#endif
    for (int64_t r = 0; r < total; ++r) {
        int64_t i = r % m, bh = r / m, b = bh / h;
        int64_t len_b = clamp_len(key_lengths, mask_kind, b, n);
        const double *qr = Q + r * d;
        const double *Kh = K + bh * n * d;
        double mu = -INFINITY;
        for (int64_t j = 0; j < n; ++j) {
            if (!key_allowed(mask_kind, i, j, len_b)) continue;
            const double *kj = Kh + j * d;
            double dot = 0.0;
            for (int64_t c = 0; c < d; ++c) dot += qr[c] * kj[c];
            if (scale * dot > mu) mu = scale * dot;
        }
        if (mu == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double Z = 0.0;
        for (int64_t j = 0; j < n; ++j) {
            if (!key_allowed(mask_kind, i, j, len_b)) continue;
            const double *kj = Kh + j * d;
            double dot = 0.0;
            for (int64_t c = 0; c < d; ++c) dot += qr[c] * kj[c];
            Z += exp(scale * dot - mu);
        }
        lse[r] = mu + log(Z);
    }
    return 0;
}

/*
 * Gradients of sum(dO * O) with respect to Q, K and V, O the attention output
 * above, dO an upstream gradient [B][h][m][d].  The pages train the model
 * (slide deck "Training Details"; primer "Training and Implementation Details")
 * but do not write the backward pass out: it is the chain rule applied to the
 * attention equation.  With p_ij the softmax weights of row i (0 for masked
 * keys) and s_ij = scale * q_i . k_j:
 *
 *   O_i   = sum_j p_ij v_j                  =>  dV_j  = sum_i p_ij dO_i
 *   dP_ij = dO_i . v_j
 *   p_i.  = softmax(s_i.)                   =>  dS_ij = p_ij (dP_ij - sum_k p_ik dP_ik)
 *   s_ij  = scale q_i . k_j                 =>  dQ_i  = scale sum_j dS_ij k_j,
 *                                               dK_j  = scale sum_i dS_ij q_i
 *
 * A row with no allowed key has output 0 whatever Q, K, V are: it contributes
 * nothing.  The work runs as two loops over the same definitions: per query row
 * (weights, dP, the row term D_i = sum_k p_ik dP_ik, dQ_i) and per key row (dV_j,
 * dK_j, recomputing p_ij and dP_ij from the saved row max, normaliser and D_i).
 * Only the (batch, head) pairs listed in bh_list are computed (all when
 * bh_list is NULL); the gradients of other pairs are left untouched.
 */
int oracle_attn_bwd(const double *Q, const double *K, const double *V, const double *dO,
                    const int32_t *key_lengths, int mask_kind, double scale,
                    int64_t B, int64_t h, int64_t m, int64_t n, int64_t d,
                    const int64_t *bh_list, int64_t nbh,
                    double *dQ, double *dK, double *dV)
{
    if (!Q || !K || !V || !dO || !dQ || !dK || !dV || B < 0 || h < 0 || m < 0 || n < 1 || d < 1) return -1;
    if (bh_list == NULL) nbh = B * h;
    double *mu = (double *)malloc(sizeof(double) * (size_t)(m > 0 ? m : 1));
    double *Z = (double *)malloc(sizeof(double) * (size_t)(m > 0 ? m : 1));
    double *D = (double *)malloc(sizeof(double) * (size_t)(m > 0 ? m : 1));
    if (!mu || !Z || !D) {
        free(mu);
        free(Z);
        free(D);
        return -1;
    }
    for (int64_t t = 0; t < nbh; ++t) {
        int64_t bh = bh_list ? bh_list[t] : t;
        int64_t len_b = clamp_len(key_lengths, mask_kind, bh / h, n);
        const double *Qh = Q + bh * m * d, *Kh = K + bh * n * d, *Vh = V + bh * n * d;
        const double *dOh = dO + bh * m * d;
        double *dQh = dQ + bh * m * d, *dKh = dK + bh * n * d, *dVh = dV + bh * n * d;

        /* per query row: softmax statistics, D_i and dQ_i */
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 8)
#endif
        for (int64_t i = 0; i < m; ++i) {
            const double *q = Qh + i * d, *g = dOh + i * d;
            double *dq = dQh + i * d;
            for (int64_t c = 0; c < d; ++c) dq[c] = 0.0;
            double mx = -INFINITY;
            for (int64_t j = 0; j < n; ++j) {
                if (!key_allowed(mask_kind, i, j, len_b)) continue;
                const double *kj = Kh + j * d;
                double dot = 0.0;
                for (int64_t c = 0; c < d; ++c) dot += q[c] * kj[c];
                if (scale * dot > mx) mx = scale * dot;
            }
            mu[i] = mx;
            Z[i] = 0.0;
            D[i] = 0.0;
            if (mx == -INFINITY) continue; /* no allowed key */
            double z = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                if (!key_allowed(mask_kind, i, j, len_b)) continue;
                const double *kj = Kh + j * d;
                double dot = 0.0;
                for (int64_t c = 0; c < d; ++c) dot += q[c] * kj[c];
                z += exp(scale * dot - mx);
            }
            Z[i] = z;
            double Di = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                if (!key_allowed(mask_kind, i, j, len_b)) continue;
                const double *kj = Kh + j * d, *vj = Vh + j * d;
                double dot = 0.0, dp = 0.0;
                for (int64_t c = 0; c < d; ++c) {
                    dot += q[c] * kj[c];
                    dp += g[c] * vj[c];
                }
                Di += exp(scale * dot - mx) / z * dp;
            }
            D[i] = Di;
            for (int64_t j = 0; j < n; ++j) {
                if (!key_allowed(mask_kind, i, j, len_b)) continue;
                const double *kj = Kh + j * d, *vj = Vh + j * d;
                double dot = 0.0, dp = 0.0;
                for (int64_t c = 0; c < d; ++c) {
                    dot += q[c] * kj[c];
                    dp += g[c] * vj[c];
                }
                double ds = exp(scale * dot - mx) / z * (dp - Di);
                for (int64_t c = 0; c < d; ++c) dq[c] += scale * ds * kj[c];
            }
        }

        /* per key row: dV_j and dK_j */
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 8)
#endif
        for (int64_t j = 0; j < n; ++j) {
            const double *k = Kh + j * d, *v = Vh + j * d;
            double *dk = dKh + j * d, *dv = dVh + j * d;
            for (int64_t c = 0; c < d; ++c) {
                dk[c] = 0.0;
                dv[c] = 0.0;
            }
            for (int64_t i = 0; i < m; ++i) {
                if (mu[i] == -INFINITY || !key_allowed(mask_kind, i, j, len_b)) continue;
                const double *q = Qh + i * d, *g = dOh + i * d;
                double dot = 0.0, dp = 0.0;
                for (int64_t c = 0; c < d; ++c) {
                    dot += q[c] * k[c];
                    dp += g[c] * v[c];
                }
                double p = exp(scale * dot - mu[i]) / Z[i];
                double ds = p * (dp - D[i]);
                for (int64_t c = 0; c < d; ++c) {
                    dv[c] += p * g[c];
                    dk[c] += scale * ds * q[c];
                }
            }
        }
    }
    free(mu);
    free(Z);
    free(D);
    return 0;
}

/* The same three functions with a restricted-attention window: keys j with
 * |i - j| <= window stay for query i when mask_kind has ORACLE_MASK_WINDOW.
 * Not reentrant (the window is held for the call); the tests call the oracle
 * from one thread. */
int oracle_attn_fwd_w(const double *Q, const double *K, const double *V, const int32_t *key_lengths,
                      int mask_kind, int64_t window, double scale, int64_t B, int64_t h, int64_t m, int64_t n,
                      int64_t d, double *out)
{
    if (window < 0) return -1;
    g_window = window;
    int rc = oracle_attn_fwd(Q, K, V, key_lengths, mask_kind, scale, B, h, m, n, d, out);
    g_window = 0;
    return rc;
}

int oracle_attn_rows_w(const double *Q, const double *K, const double *V, const int32_t *key_lengths,
                       int mask_kind, int64_t window, double scale, int64_t B, int64_t h, int64_t m, int64_t n,
                       int64_t d, const int64_t *rows, int64_t nrows, double *out)
{
    if (window < 0) return -1;
    g_window = window;
    int rc = oracle_attn_rows(Q, K, V, key_lengths, mask_kind, scale, B, h, m, n, d, rows, nrows, out);
    g_window = 0;
    return rc;
}

int oracle_attn_lse_w(const double *Q, const double *K, const int32_t *key_lengths, int mask_kind,
                      int64_t window, double scale, int64_t B, int64_t h, int64_t m, int64_t n, int64_t d,
                      double *lse)
{
    if (window < 0) return -1;
    g_window = window;
    int rc = oracle_attn_lse(Q, K, key_lengths, mask_kind, scale, B, h, m, n, d, lse);
    g_window = 0;
    return rc;
}

