/*
 * CPU oracle for the paged KV-cache composition -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this file's library.  The CUDA library never calls it and shares no
 * code, header or table with it.
 *
 * What it computes is the plain definition, in double precision:
 *   1. the slot-mapped cache write ("ReshapeAndCache->PagedAttention
 *      composition at real dims", What changed; the review asks that each
 *      token's slot come from the block table), as a bit copy;
 *   2. grouped-query causal softmax attention read back through a per-request
 *      block table (same page, What changed: Dh=256, Hq=8, Hkv=2, page 16,
 *      shuffled table), for full prefill, suffix prefill and single-query
 *      decode ("stabilize direct paged CK attention for bitwise R/R",
 *      Additional checks: full and suffix execution, causal/LSE vs decode).
 *
 * Readings where the pages are silent:
 *   - query head h reads KV head h / (Hq/Hkv) (the composition page gives
 *     only Hq=8, Hkv=2);
 *   - seq_lens[b] counts the new tokens, so query i of request b sits at
 *     position L_b - q_b + i and may see keys 0..that position (the bitwise
 *     R/R page's Operator benchmarks quote "Q128, KV7168" beside "Q1,
 *     KV7168"; its Additional checks name full and suffix execution);
 *   - scores are scale * q.k with the fp32 scale widened to double;
 *   - LSE is the natural log of the sum of exp(scores), scale included (the
 *     bitwise R/R page's Additional checks name LSE without a formula).
 * There is no blocking, tiling, online rescaling or chunking here: scores
 * are materialised, the maximum taken, then the normalised sum formed.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define PAO_BLOCK_SIZE 16

static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Cache write.  Token i with slot s >= 0 lands in block s / 16 at offset
 * s % 16, one Dh-long row per KV head, for K and for V.  A negative slot
 * is a padding token and is skipped.  Returns 0, or 1 + the index of the
 * first token whose slot is past the pool (that token is not written).
 * Element offsets are 64-bit: pools may exceed 2**31 elements.
 */
int64_t pao_reshape_and_cache(const uint16_t *key, int64_t key_tok_stride,
                              const uint16_t *value, int64_t value_tok_stride,
                              int64_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                              uint16_t *k_pool, uint16_t *v_pool, int64_t num_blocks,
                              int64_t block_stride, int64_t token_stride, int64_t head_stride,
                              const int64_t *slot_mapping)
{
    int64_t first_bad = 0;
    for (int64_t i = 0; i < num_tokens; ++i) {
        int64_t s = slot_mapping[i];
        if (s < 0)
            continue;
        if (s >= num_blocks * PAO_BLOCK_SIZE) {
            if (!first_bad)
                first_bad = i + 1;
            continue;
        }
        int64_t blk = s / PAO_BLOCK_SIZE, off = s % PAO_BLOCK_SIZE;
        for (int32_t h = 0; h < num_kv_heads; ++h) {
            int64_t dst = blk * block_stride + off * token_stride + (int64_t)h * head_stride;
            const uint16_t *ks = key + i * key_tok_stride + (int64_t)h * head_dim;
            const uint16_t *vs = value + i * value_tok_stride + (int64_t)h * head_dim;
            for (int32_t d = 0; d < head_dim; ++d) {
                k_pool[dst + d] = ks[d];
                v_pool[dst + d] = vs[d];
            }
        }
    }
    return first_bad;
}

/* Which request owns flattened query token t (query_start_loc is sorted). */
static int32_t owner_of(const int32_t *qsl, int32_t num_seqs, int64_t t)
{
    int32_t lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
        int32_t mid = (lo + hi + 1) / 2;
        if (qsl[mid] <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

/*
 * Paged attention.  For each requested query token (rows[] if given, else
 * all tokens 0..num_q_tokens-1) and each query head, writes
 *   out[r][h][d] = sum_j w_j V_j[d],  w_j = exp(s_j - m) / sum_k exp(s_k - m),
 *   lse[r][h]    = m + log(sum_k exp(s_k - m)),
 * over keys j = 0..pos, with K_j/V_j fetched from block
 * block_tables[b][j/16] at offset j%16.  out is [R][Hq][Dh] doubles and lse
 * [R][Hq] doubles, R = num_rows.  Returns 0, or 1 + the flat index of the
 * first (row, head) whose metadata was unusable (that row is NaN).
 */
int64_t pao_paged_attention(const uint16_t *q, int64_t q_tok_stride, int32_t num_q_heads,
                            const uint16_t *k_pool, const uint16_t *v_pool, int64_t num_blocks,
                            int64_t block_stride, int64_t token_stride, int64_t head_stride,
                            int32_t num_kv_heads, int32_t head_dim,
                            const int32_t *block_tables, int32_t max_blocks_per_seq,
                            const int32_t *seq_lens, const int32_t *query_start_loc,
                            int32_t num_seqs, float scale, const int64_t *rows, int64_t num_rows,
                            double *out, double *lse, int32_t num_threads)
{
    const int32_t group = num_q_heads / num_kv_heads;
    const double sc = (double)scale;
    int64_t first_bad = 0;
#ifdef _OPENMP
    if (num_threads > 0)
        omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif
    const int64_t work = num_rows * (int64_t)num_q_heads;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t w = 0; w < work; ++w) {
        const int64_t r = w / num_q_heads;
        const int32_t h = (int32_t)(w % num_q_heads);
        const int64_t t = rows ? rows[r] : r;
        double *o = out + w * head_dim;
        const int32_t b = owner_of(query_start_loc, num_seqs, t);
        const int64_t qn = (int64_t)query_start_loc[b + 1] - query_start_loc[b];
        const int64_t L = seq_lens[b];
        const int64_t pos = L - qn + (t - query_start_loc[b]);
        const int32_t g = h / group;
        int bad = (qn < 0 || L < qn || pos < 0 || L > (int64_t)max_blocks_per_seq * PAO_BLOCK_SIZE);
        double *s = NULL;
        if (!bad) {
            s = (double *)malloc(sizeof(double) * (size_t)(pos + 1));
            bad = (s == NULL);
        }
        /* scores s_j = scale * sum_d q[d] k_j[d] */
        const uint16_t *qrow = q + t * q_tok_stride + (int64_t)h * head_dim;
        for (int64_t j = 0; !bad && j <= pos; ++j) {
            int64_t blk = block_tables[(int64_t)b * max_blocks_per_seq + j / PAO_BLOCK_SIZE];
            if (blk < 0 || blk >= num_blocks) {
                bad = 1;
                break;
            }
            const uint16_t *krow = k_pool + blk * block_stride + (j % PAO_BLOCK_SIZE) * token_stride
                                   + (int64_t)g * head_stride;
            double dot = 0.0;
            for (int32_t d = 0; d < head_dim; ++d)
                dot += bf16_bits_to_double(qrow[d]) * bf16_bits_to_double(krow[d]);
            s[j] = sc * dot;
        }
        if (bad) {
            for (int32_t d = 0; d < head_dim; ++d)
                o[d] = NAN;
            lse[w] = NAN;
            free(s);
#pragma omp critical
            if (!first_bad || w + 1 < first_bad)
                first_bad = w + 1;
            continue;
        }
        double m = -INFINITY;
        for (int64_t j = 0; j <= pos; ++j)
            if (s[j] > m)
                m = s[j];
        double denom = 0.0;
        for (int64_t j = 0; j <= pos; ++j)
            denom += exp(s[j] - m);
        for (int32_t d = 0; d < head_dim; ++d)
            o[d] = 0.0;
        for (int64_t j = 0; j <= pos; ++j) {
            int64_t blk = block_tables[(int64_t)b * max_blocks_per_seq + j / PAO_BLOCK_SIZE];
            const uint16_t *vrow = v_pool + blk * block_stride + (j % PAO_BLOCK_SIZE) * token_stride
                                   + (int64_t)g * head_stride;
            double wj = exp(s[j] - m) / denom;
            for (int32_t d = 0; d < head_dim; ++d)
                o[d] += wj * bf16_bits_to_double(vrow[d]);
        }
        lse[w] = m + log(denom);
        free(s);
    }
    return first_bad;
}

int32_t pao_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
