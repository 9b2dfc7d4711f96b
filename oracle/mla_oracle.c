/*
 * Oracle for the MLA latent-cache decode step: plain, slow, fp64, CPU only.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this file: it is used by the tests, by the smoke check and by the
 * CPU-baseline leg of the benchmark.  It shares no code, header, table or
 * helper with the CUDA library; the two meet only at the seeded inputs.
 *
 * What is computed, and where it is stated:
 *
 *  - Absorbed-form decode.  Each head's query has already been projected into
 *    the latent space, so every head attends directly over the one shared
 *    576-wide latent row of each cached token
 *      [dp-attention-expert-parallel-mla-kv-replication (inferenceinterviews.com),
 *       "A strong answer", paragraph on the absorbed form].
 *  - The cached row is 512 kv_c values followed by 64 k_rope values; the 64
 *    rope dims are MQA-style, shared by all 128 heads, so all 576 dims feed
 *    every head's score
 *      [MLA 的 TP 切分：为什么 8 张 GPU 存了同一份 KV cache (10100.com),
 *       section 一 and section 2.2 "三个事实", section 3.1 cache picture:
 *       elements 0-511 = kv_c, 512-575 = k_rope, layout [NB, BS, 576]].
 *  - The value vector is the 512-wide kv_c itself (v_head_dim = kv_lora_rank)
 *      [DP 与 DPA 的区别 (chengxuchu.com), "MLA：KV 是一份共享 latent" code note].
 *  - Softmax attention: the plain textbook definition, written out
 *        s_t   = scale * sum_{d<576} q[h][d] * row_t[d]
 *        m     = max_t s_t,  w_t = exp(s_t - m),  Z = sum_t w_t
 *        out_j = sum_t (w_t / Z) * row_t[j]       for j < 512
 *        lse   = m + ln Z
 *    The pages never print this equation; it is the plainest reading of the
 *    absorbed form with K = the full 576-wide row and V = its first 512 dims.
 *  - Paging: token t of request b lives in block block_table[b][t / BS] at row
 *    t mod BS  [MLA 的 TP 切分 (10100.com), section 3.1, MLAAttentionSpec with
 *    block_size from the cache config; layout NL x NB x BS x HS].
 *  - Append: the new 576-wide kv_a_proj_with_mqa row of a token is stored
 *    byte-for-byte at its slot  [MLA 的 TP 切分 (10100.com), section 2.2].
 *  - Split combine: partial results over disjoint token ranges, each carrying
 *    its log-sum-exp, merge as  out = sum_s e^{lse_s - M} o_s / sum_s e^{lse_s - M},
 *    lse = M + ln sum_s e^{lse_s - M}.  This is the same softmax definition
 *    regrouped over the ranges; it is not on the pages.
 *
 * Inputs in bfloat16 are passed as their raw 16-bit patterns and widened
 * exactly (bits << 16) to binary32, then to binary64.  All arithmetic is fp64.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>

#define ORACLE_ROW 576      /* 512 kv_c + 64 k_rope */
#define ORACLE_VDIM 512     /* kv_lora_rank: the value width */

static double bf16_to_f64(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Location of logical token t of request b, or NULL if the table is bad. */
static const uint16_t *token_row(const uint16_t *cache, int64_t num_blocks, int32_t block_size,
                                 const int32_t *block_table, int32_t max_blocks_per_seq,
                                 int32_t b, int32_t t) {
    int32_t blk = block_table[(int64_t)b * max_blocks_per_seq + t / block_size];
    if (blk < 0 || (int64_t)blk >= num_blocks) return NULL;
    return cache + ((int64_t)blk * block_size + (t % block_size)) * ORACLE_ROW;
}

/*
 * Attention of every (request, head) over the token range [t_begin[b], t_end[b]).
 * out: [batch][num_heads][512] fp64;  lse: [batch][num_heads] fp64 (natural log).
 * An empty range gives out = 0 and lse = -inf.  Returns 0, or -1 on a bad
 * block-table entry, -2 on a bad range.
 */
int oracle_decode_range(const uint16_t *q, const uint16_t *cache, int64_t num_blocks,
                        int32_t block_size, const int32_t *block_table,
                        int32_t max_blocks_per_seq, const int32_t *t_begin,
                        const int32_t *t_end, int32_t batch, int32_t num_heads,
                        double softmax_scale, double *out, double *lse) {
    for (int32_t b = 0; b < batch; ++b) {
        if (t_begin[b] < 0 || t_end[b] < t_begin[b] ||
            (int64_t)t_end[b] > (int64_t)max_blocks_per_seq * block_size)
            return -2;
        for (int32_t t = t_begin[b]; t < t_end[b]; ++t)
            if (!token_row(cache, num_blocks, block_size, block_table, max_blocks_per_seq, b, t))
                return -1;
    }
    int64_t pairs = (int64_t)batch * num_heads;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < pairs; ++bh) {
        int32_t b = (int32_t)(bh / num_heads);
        const uint16_t *qh = q + bh * ORACLE_ROW;
        double *o = out + bh * ORACLE_VDIM;
        int32_t n = t_end[b] - t_begin[b];
        for (int j = 0; j < ORACLE_VDIM; ++j) o[j] = 0.0;
        if (n == 0) {
            lse[bh] = -INFINITY;
            continue;
        }
        double qd[ORACLE_ROW];
        for (int d = 0; d < ORACLE_ROW; ++d) qd[d] = bf16_to_f64(qh[d]);
        double *s = (double *)malloc(sizeof(double) * (size_t)n);
        /* scores over all 576 dims */
        double m = -INFINITY;
        for (int32_t i = 0; i < n; ++i) {
            const uint16_t *row = token_row(cache, num_blocks, block_size, block_table,
                                            max_blocks_per_seq, b, t_begin[b] + i);
            double acc = 0.0;
            for (int d = 0; d < ORACLE_ROW; ++d) acc += qd[d] * bf16_to_f64(row[d]);
            s[i] = softmax_scale * acc;
            if (s[i] > m) m = s[i];
        }
        /* normaliser */
        double z = 0.0;
        for (int32_t i = 0; i < n; ++i) z += exp(s[i] - m);
        /* weighted sum of the kv_c part (first 512 dims) */
        for (int32_t i = 0; i < n; ++i) {
            const uint16_t *row = token_row(cache, num_blocks, block_size, block_table,
                                            max_blocks_per_seq, b, t_begin[b] + i);
            double p = exp(s[i] - m) / z;
            for (int j = 0; j < ORACLE_VDIM; ++j) o[j] += p * bf16_to_f64(row[j]);
        }
        lse[bh] = m + log(z);
        free(s);
    }
    return 0;
}

/* Full-context decode: every request attends over tokens [0, seq_lens[b]). */
int oracle_decode(const uint16_t *q, const uint16_t *cache, int64_t num_blocks,
                  int32_t block_size, const int32_t *block_table, int32_t max_blocks_per_seq,
                  const int32_t *seq_lens, int32_t batch, int32_t num_heads,
                  double softmax_scale, double *out, double *lse) {
    int32_t *zeros = (int32_t *)calloc((size_t)(batch > 0 ? batch : 1), sizeof(int32_t));
    int rc = oracle_decode_range(q, cache, num_blocks, block_size, block_table,
                                 max_blocks_per_seq, zeros, seq_lens, batch, num_heads,
                                 softmax_scale, out, lse);
    free(zeros);
    return rc;
}

/*
 * The attention weights p_t of one (request, head) over [0, seq_len): lets the
 * tests check that each softmax row sums to one.  p must hold seq_len doubles.
 */
int oracle_probs(const uint16_t *q, const uint16_t *cache, int64_t num_blocks,
                 int32_t block_size, const int32_t *block_table, int32_t max_blocks_per_seq,
                 const int32_t *seq_lens, int32_t num_heads, int32_t b, int32_t h,
                 double softmax_scale, double *p) {
    int32_t n = seq_lens[b];
    const uint16_t *qh = q + ((int64_t)b * num_heads + h) * ORACLE_ROW;
    double m = -INFINITY;
    for (int32_t t = 0; t < n; ++t) {
        const uint16_t *row = token_row(cache, num_blocks, block_size, block_table,
                                        max_blocks_per_seq, b, t);
        if (!row) return -1;
        double acc = 0.0;
        for (int d = 0; d < ORACLE_ROW; ++d) acc += bf16_to_f64(qh[d]) * bf16_to_f64(row[d]);
        p[t] = softmax_scale * acc;
        if (p[t] > m) m = p[t];
    }
    double z = 0.0;
    for (int32_t t = 0; t < n; ++t) {
        p[t] = exp(p[t] - m);
        z += p[t];
    }
    for (int32_t t = 0; t < n; ++t) p[t] /= z;
    return 0;
}

/*
 * Append: row i of kv_new (576 bf16 = 1152 bytes) is copied to slot
 * slot_mapping[i], i.e. block slot / BS, row slot mod BS.  Slot -1 is skipped.
 * Returns 0, or -1 if any slot is outside [-1, num_blocks * block_size) (and
 * then nothing is written).
 */
int oracle_append(const uint16_t *kv_new, const int64_t *slot_mapping, int64_t num_tokens,
                  uint16_t *cache, int64_t num_blocks, int32_t block_size) {
    int64_t slots = num_blocks * (int64_t)block_size;
    for (int64_t i = 0; i < num_tokens; ++i)
        if (slot_mapping[i] < -1 || slot_mapping[i] >= slots) return -1;
    for (int64_t i = 0; i < num_tokens; ++i) {
        int64_t s = slot_mapping[i];
        if (s < 0) continue;
        int64_t blk = s / block_size, row = s % block_size;
        memcpy(cache + (blk * block_size + row) * ORACLE_ROW, kv_new + i * ORACLE_ROW,
               ORACLE_ROW * sizeof(uint16_t));
    }
    return 0;
}

/*
 * Merge of split partials.  Request b owns partial rows
 * [split_offsets[b], split_offsets[b+1]); each row w holds o_partial[w][h][512]
 * (already normalised by its own sum) and lse_partial[w][h].
 * out[b][h][j] = sum_w e^{lse_w - M} o_w / sum_w e^{lse_w - M}; lse = M + ln sum.
 * Partials with lse = -inf (empty ranges) carry zero weight; a request whose
 * partials are all empty gives out = 0, lse = -inf.
 */
void oracle_combine(const double *o_partial, const double *lse_partial,
                    const int32_t *split_offsets, int32_t batch, int32_t num_heads,
                    double *out, double *lse) {
    for (int32_t b = 0; b < batch; ++b) {
        for (int32_t h = 0; h < num_heads; ++h) {
            double *o = out + ((int64_t)b * num_heads + h) * ORACLE_VDIM;
            double m = -INFINITY;
            for (int32_t w = split_offsets[b]; w < split_offsets[b + 1]; ++w) {
                double l = lse_partial[(int64_t)w * num_heads + h];
                if (l > m) m = l;
            }
            for (int j = 0; j < ORACLE_VDIM; ++j) o[j] = 0.0;
            if (m == -INFINITY) {
                lse[(int64_t)b * num_heads + h] = -INFINITY;
                continue;
            }
            double z = 0.0;
            for (int32_t w = split_offsets[b]; w < split_offsets[b + 1]; ++w) {
                double l = lse_partial[(int64_t)w * num_heads + h];
                if (l == -INFINITY) continue;
                double e = exp(l - m);
                z += e;
                const double *ow = o_partial + ((int64_t)w * num_heads + h) * ORACLE_VDIM;
                for (int j = 0; j < ORACLE_VDIM; ++j) o[j] += e * ow[j];
            }
            for (int j = 0; j < ORACLE_VDIM; ++j) o[j] /= z;
            lse[(int64_t)b * num_heads + h] = m + log(z);
        }
    }
}

/* Threads the OpenMP runtime will use; lets the baseline report its core count. */
int oracle_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
