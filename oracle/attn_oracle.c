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
 * Readings of the pages taken here (each one is listed in the design doc):
 *  - key padding is trailing: key j of batch b is masked iff j >= len_b, the
 *    same for every head; len_b is clamped to [0, n]; query rows are never
 *    masked by padding;
 *  - causal masks key j for query i iff j > i (queries and keys share
 *    positions; the library rejects causal with m != n);
 *  - a query row with no allowed key has output 0 (the formula gives 0/0);
 *  - the scale is an argument (1/sqrt(d_k) in the formula; the pages' worked
 *    example needs other values).
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

/* M_ij == 0 (allowed) or -inf (masked): deep reading §04, §03 "Decoder layer". */
static int key_allowed(int mask_kind, int64_t i, int64_t j, int64_t len_b)
{
    if ((mask_kind & ORACLE_MASK_CAUSAL) && j > i) return 0;
    if ((mask_kind & ORACLE_MASK_KEY_PADDING) && j >= len_b) return 0;
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
