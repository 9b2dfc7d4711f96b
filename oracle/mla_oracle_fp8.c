/*
 * Oracle for the FP8 latent cache: plain, slow, fp64, CPU only.
 *
 * TEST INFRASTRUCTURE ONLY, under the same rules as mla_oracle.c: nothing on
 * the product path may include, link or call this file, and it shares no
 * code, header, table or helper with the CUDA library.
 *
 * What the pages fix: an FP8 latent cache stores one byte per latent element,
 * 576 bytes per token per layer (512 kv_c + 64 k_rope)
 *   [MLA 的 TP 切分 (10100.com), opening paragraph (32 KB -> 576 bytes per
 *    token per layer) and section 5.1 (576 bytes in FP8 per token per layer)].
 * The pages name no 8-bit format, no scale and no rounding.  The readings
 * taken here (the plainest ones consistent with 576 bytes per token):
 *  - The format is OCP FP8 E4M3: 1 sign bit, 4 exponent bits with bias 7,
 *    3 mantissa bits, no infinities, S.1111.111 is NaN, the largest finite
 *    magnitude is 448, subnormals are 2^-6 * m/8.
 *  - One scale per layer, kv_scale > 0 (1 when unused): a stored code c
 *    stands for value(c) * kv_scale.  There is no per-token scale, so a row
 *    stays 576 bytes.
 *  - A new bf16 row element x is stored as the code nearest to
 *    y = fp32(x) * fp32(1 / kv_scale) (both roundings in fp32, the
 *    precision the product is formed in), ties to the even code, magnitudes
 *    above 448 saturating to 448, NaN to NaN (code 0x7F).
 * Decode over an FP8 cache is the same softmax attention as mla_oracle.c
 * (absorbed form, K = the 576-wide row, V = its first 512 dims), with every
 * row element value(code) * kv_scale.  All arithmetic is fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define FP8_ROW 576
#define FP8_VDIM 512

/* Value of an E4M3 code, from the format's definition. */
double oracle_e4m3_value(uint8_t code) {
    const int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    const double mag = e == 0 ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* The E4M3 code for y: the nearest finite value (ties: the even code),
 * saturating to +-448; NaN gives 0x7F.  Brute force over the 127 finite
 * non-negative codes, whose values increase with the code. */
uint8_t oracle_e4m3_encode(float y) {
    if (isnan(y)) return 0x7F;
    const int neg = signbit(y) ? 1 : 0;
    const double a = fabs((double)y);
    uint8_t best = 0x7E;
    if (a < 448.0) {
        double best_err = INFINITY;
        for (int c = 0; c <= 0x7E; ++c) {
            const double err = fabs(oracle_e4m3_value((uint8_t)c) - a);
            if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
                best_err = err;
                best = (uint8_t)c;
            }
        }
    }
    return (uint8_t)(neg ? (0x80 | best) : best);
}

static float bf16_bits_to_f32(uint16_t bits) {
    const uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Quantise n bf16 values: out[i] = encode(fp32(x_i) * fp32(1 / kv_scale)). */
void oracle_quantize_rows(const uint16_t *bf16, int64_t n, float kv_scale, uint8_t *out) {
    const float inv = 1.0f / kv_scale;
    for (int64_t i = 0; i < n; ++i) {
        volatile float y = bf16_bits_to_f32(bf16[i]) * inv;  /* one fp32 rounding */
        out[i] = oracle_e4m3_encode(y);
    }
}

/* Store each new bf16 row, quantised, at its slot of the FP8 cache
 * [num_slots][576] bytes; slot -1 is skipped.  Returns 0, or -1 if a slot is
 * outside [-1, num_slots). */
int oracle_append_fp8(const uint16_t *kv_new, const int64_t *slot_mapping, int64_t num_tokens,
                      float kv_scale, uint8_t *cache, int64_t num_slots) {
    for (int64_t i = 0; i < num_tokens; ++i)
        if (slot_mapping[i] < -1 || slot_mapping[i] >= num_slots) return -1;
    for (int64_t i = 0; i < num_tokens; ++i) {
        if (slot_mapping[i] < 0) continue;
        oracle_quantize_rows(kv_new + i * FP8_ROW, FP8_ROW, kv_scale,
                             cache + slot_mapping[i] * FP8_ROW);
    }
    return 0;
}

/*
 * Decode over an FP8 cache [num_blocks][block_size][576] bytes: for every
 * request b (context seq_lens[b]) and head h,
 *     row_t[d] = value(code) * kv_scale,
 *     s_t = softmax_scale * sum_{d<576} q[b,h,d] row_t[d],
 *     out[b,h,j] = sum_t softmax(s)_t row_t[j]  (j < 512),  lse = log sum_t e^{s_t}.
 * q is bf16 (raw bits).  An empty context gives out = 0, lse = -inf.
 * Returns 0, or -1 on a block-table entry outside the pool.
 */
int oracle_decode_fp8(const uint16_t *q, const uint8_t *cache, double kv_scale,
                      int64_t num_blocks, int32_t block_size, const int32_t *block_table,
                      int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t batch,
                      int32_t num_heads, double softmax_scale, double *out, double *lse) {
    for (int32_t b = 0; b < batch; ++b)
        for (int32_t t = 0; t < seq_lens[b]; t += block_size) {
            const int32_t blk = block_table[(int64_t)b * max_blocks_per_seq + t / block_size];
            if (blk < 0 || (int64_t)blk >= num_blocks) return -1;
        }
    /* the stored value of every code, scaled: row element = value(code) * kv_scale */
    double val[256];
    for (int c = 0; c < 256; ++c) val[c] = oracle_e4m3_value((uint8_t)c) * kv_scale;
    const int64_t pairs = (int64_t)batch * num_heads;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < pairs; ++bh) {
        const int32_t b = (int32_t)(bh / num_heads);
        const int32_t L = seq_lens[b];
        const uint16_t *qh = q + bh * FP8_ROW;
        double *o = out + bh * FP8_VDIM;
        for (int j = 0; j < FP8_VDIM; ++j) o[j] = 0.0;
        if (L <= 0) {
            lse[bh] = -INFINITY;
            continue;
        }
        double qd[FP8_ROW];
        for (int d = 0; d < FP8_ROW; ++d) qd[d] = (double)bf16_bits_to_f32(qh[d]);
        double *s = (double *)malloc(sizeof(double) * (size_t)L);
        /* scores over all 576 dims */
        double m = -INFINITY;
        for (int32_t t = 0; t < L; ++t) {
            const int32_t blk = block_table[(int64_t)b * max_blocks_per_seq + t / block_size];
            const uint8_t *row = cache + ((int64_t)blk * block_size + t % block_size) * FP8_ROW;
            double acc = 0.0;
            for (int d = 0; d < FP8_ROW; ++d) acc += qd[d] * val[row[d]];
            s[t] = softmax_scale * acc;
            if (s[t] > m) m = s[t];
        }
        /* normaliser, then the weighted sum of the kv_c part (first 512 dims) */
        double z = 0.0;
        for (int32_t t = 0; t < L; ++t) z += exp(s[t] - m);
        for (int32_t t = 0; t < L; ++t) {
            const int32_t blk = block_table[(int64_t)b * max_blocks_per_seq + t / block_size];
            const uint8_t *row = cache + ((int64_t)blk * block_size + t % block_size) * FP8_ROW;
            const double p = exp(s[t] - m) / z;
            for (int j = 0; j < FP8_VDIM; ++j) o[j] += p * val[row[j]];
        }
        lse[bh] = m + log(z);
        free(s);
    }
    return 0;
}
