// CUDA-core MLA decode: the first correct GPU path (fp32 FMA, no tensor cores).
//
// CTA (range p, head group g) walks the request segments of plan range p for
// 16 heads.  Per tile of 32 tokens: the paged latent rows are staged in shared
// memory, each of the 16 heads scores every row over all 576 dims (512 kv_c +
// 64 shared k_rope), an online softmax (running max / sum in registers,
// 16-lane shuffles) rescales the fp32 output, and the output accumulates the
// 512 kv_c dims weighted by the probabilities.  Absorbed-form decode over the
// shared latent [dp-attention-expert-parallel-mla-kv-replication
// (inferenceinterviews.com), "A strong answer"]; value = kv_c
// [DP 与 DPA 的区别 (chengxuchu.com), "MLA：KV 是一份共享 latent"].
#include "common.cuh"

namespace mla {

constexpr int kSimtHeads = 16;     // heads per CTA
constexpr int kSimtTile = 32;      // tokens per tile (= plan unit)
constexpr int kSimtThreads = 256;  // 16 threads per head
constexpr int kRowPad = kRow + 8;  // bf16 elements per staged row (bank spread)

struct SimtSmem {
  float q[kSimtHeads][kRow];
  __nv_bfloat16 rows[kSimtTile][kRowPad];
  float p[kSimtHeads][kSimtTile];
};

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__global__ void __launch_bounds__(kSimtThreads) decode_simt_kernel(
    const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ cache,
    int64_t num_blocks, int32_t block_size, const int32_t *__restrict__ block_table,
    int32_t max_blocks_per_seq, int32_t batch, float scale_log2, __nv_bfloat16 *__restrict__ out,
    float *__restrict__ lse, void *ws, int32_t max_ranges, int32_t *dev_status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SimtSmem &sm = *reinterpret_cast<SimtSmem *>(smem_raw);
  PlanView v = plan_view(ws, batch, kHeads, max_ranges);
  const int tid = threadIdx.x;
  const int hl = tid / 16, sub = tid % 16;
  const int h = blockIdx.y * kSimtHeads + hl;
  const int p = blockIdx.x;

  // requests with no context: out = 0, lse = -inf
  for (int b = p; b < batch; b += gridDim.x) {
    if (v.seq_len[b] != 0) continue;
    uint4 *o = (uint4 *)(out + ((int64_t)b * kHeads + h) * kVDim);
    for (int k = sub; k < kVDim / 8; k += 16) o[k] = make_uint4(0, 0, 0, 0);
    if (lse && sub == 0) lse[(int64_t)b * kHeads + h] = -INFINITY;
  }

  const int32_t U = v.hdr->total_units, P = v.hdr->num_ranges;
  if (p >= P) return;
  const int32_t r0 = range_begin(p, U, P), r1 = range_begin(p + 1, U, P);

  for (int b = v.range_first[p]; b < batch && v.unit_prefix[b] < r1; ++b) {
    const int32_t Ub = v.unit_prefix[b], Ue = v.unit_prefix[b + 1];
    if (Ue == Ub) continue;
    const int32_t u0 = max(r0, Ub), u1 = min(r1, Ue);
    if (u0 >= u1) continue;
    const int32_t L = v.seq_len[b];
    const int32_t t_begin = (u0 - Ub) * kSimtTile;
    const int32_t t_end = min((u1 - Ub) * kSimtTile, L);
    const bool split = range_of(Ub, U, P) != range_of(Ue - 1, U, P);

    __syncthreads();  // previous segment done with q / rows
    for (int k = tid; k < kSimtHeads * kRow / 2; k += kSimtThreads) {
      const int hh = k / (kRow / 2), d2 = k % (kRow / 2);
      const uint32_t w = reinterpret_cast<const uint32_t *>(
          q + ((int64_t)b * kHeads + blockIdx.y * kSimtHeads + hh) * kRow)[d2];
      sm.q[hh][2 * d2] = bf16lo(w);
      sm.q[hh][2 * d2 + 1] = bf16hi(w);
    }
    float m = -INFINITY, l = 0.f;
    float acc[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) acc[j] = 0.f;

    for (int t0 = t_begin; t0 < t_end; t0 += kSimtTile) {
      const int n = min(kSimtTile, t_end - t0);
      __syncthreads();  // rows / p of the previous tile consumed
      for (int k = tid; k < n * (kRow / 8); k += kSimtThreads) {
        const int r = k / (kRow / 8), c = k % (kRow / 8);
        const int t = t0 + r;
        const int32_t blk = block_table[(int64_t)b * max_blocks_per_seq + t / block_size];
        uint4 val = make_uint4(0, 0, 0, 0);
        if (blk >= 0 && (int64_t)blk < num_blocks) {
          val = reinterpret_cast<const uint4 *>(
              cache + ((int64_t)blk * block_size + t % block_size) * kRow)[c];
        } else if (c == 0) {
          report(dev_status, MLA_ERR_DEVICE_RANGE);
        }
        *reinterpret_cast<uint4 *>(&sm.rows[r][8 * c]) = val;
      }
      __syncthreads();
      // scores of tokens sub and sub + 16 for head hl, in log2 units
      float s[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int r = sub + 16 * i;
        float a = 0.f;
        if (r < n) {
          const uint4 *row = reinterpret_cast<const uint4 *>(&sm.rows[r][0]);
          const float4 *qq = reinterpret_cast<const float4 *>(&sm.q[hl][0]);
#pragma unroll 4
          for (int c = 0; c < kRow / 8; ++c) {
            const uint4 w = row[c];
            const float4 qa = qq[2 * c], qb = qq[2 * c + 1];
            a = fmaf(qa.x, bf16lo(w.x), a); a = fmaf(qa.y, bf16hi(w.x), a);
            a = fmaf(qa.z, bf16lo(w.y), a); a = fmaf(qa.w, bf16hi(w.y), a);
            a = fmaf(qb.x, bf16lo(w.z), a); a = fmaf(qb.y, bf16hi(w.z), a);
            a = fmaf(qb.z, bf16lo(w.w), a); a = fmaf(qb.w, bf16hi(w.w), a);
          }
          s[i] = a * scale_log2;
        } else {
          s[i] = -INFINITY;
        }
      }
      float tmax = fmaxf(s[0], s[1]);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o, 16));
      const float m_new = fmaxf(m, tmax);
      const float alpha = exp2f(m - m_new);
      const float p0 = exp2f(s[0] - m_new), p1 = exp2f(s[1] - m_new);
      float ps = p0 + p1;
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o, 16);
      l = l * alpha + ps;
      m = m_new;
      sm.p[hl][sub] = p0;
      sm.p[hl][sub + 16] = p1;
#pragma unroll
      for (int j = 0; j < 32; ++j) acc[j] *= alpha;
      __syncthreads();
      for (int r = 0; r < n; ++r) {
        const float pr = sm.p[hl][r];
        const uint4 *row = reinterpret_cast<const uint4 *>(&sm.rows[r][sub * 32]);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 w = row[c];
          acc[8 * c + 0] = fmaf(pr, bf16lo(w.x), acc[8 * c + 0]);
          acc[8 * c + 1] = fmaf(pr, bf16hi(w.x), acc[8 * c + 1]);
          acc[8 * c + 2] = fmaf(pr, bf16lo(w.y), acc[8 * c + 2]);
          acc[8 * c + 3] = fmaf(pr, bf16hi(w.y), acc[8 * c + 3]);
          acc[8 * c + 4] = fmaf(pr, bf16lo(w.z), acc[8 * c + 4]);
          acc[8 * c + 5] = fmaf(pr, bf16hi(w.z), acc[8 * c + 5]);
          acc[8 * c + 6] = fmaf(pr, bf16lo(w.w), acc[8 * c + 6]);
          acc[8 * c + 7] = fmaf(pr, bf16hi(w.w), acc[8 * c + 7]);
        }
      }
    }
    const float inv = 1.f / l;
    const float lse_val = (m + log2f(l)) * 0.69314718055994531f;
    if (!split) {
      uint4 *o = (uint4 *)(out + ((int64_t)b * kHeads + h) * kVDim + sub * 32);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        __nv_bfloat162 x0 = __floats2bfloat162_rn(acc[8 * c + 0] * inv, acc[8 * c + 1] * inv);
        __nv_bfloat162 x1 = __floats2bfloat162_rn(acc[8 * c + 2] * inv, acc[8 * c + 3] * inv);
        __nv_bfloat162 x2 = __floats2bfloat162_rn(acc[8 * c + 4] * inv, acc[8 * c + 5] * inv);
        __nv_bfloat162 x3 = __floats2bfloat162_rn(acc[8 * c + 6] * inv, acc[8 * c + 7] * inv);
        uint4 w;
        w.x = *reinterpret_cast<uint32_t *>(&x0);
        w.y = *reinterpret_cast<uint32_t *>(&x1);
        w.z = *reinterpret_cast<uint32_t *>(&x2);
        w.w = *reinterpret_cast<uint32_t *>(&x3);
        o[c] = w;
      }
      if (lse && sub == 0) lse[(int64_t)b * kHeads + h] = lse_val;
    } else {
      const int slot = partial_slot(p, U, P, Ub);
      float4 *o = (float4 *)(v.o_part + ((int64_t)slot * kHeads + h) * kVDim + sub * 32);
#pragma unroll
      for (int c = 0; c < 8; ++c)
        o[c] = make_float4(acc[4 * c] * inv, acc[4 * c + 1] * inv, acc[4 * c + 2] * inv,
                           acc[4 * c + 3] * inv);
      if (sub == 0) v.lse_part[(int64_t)slot * kHeads + h] = lse_val;
    }
  }
}

int simt_unit_tokens() { return kSimtTile; }

cudaError_t launch_decode_simt(const void *q, const void *cache, int64_t num_blocks,
                               int32_t block_size, const int32_t *block_table,
                               int32_t max_blocks_per_seq, int32_t batch, float softmax_scale,
                               void *out, float *lse, void *ws, int32_t max_ranges,
                               int32_t *dev_status, cudaStream_t stream) {
  const size_t smem = sizeof(SimtSmem);
  cudaError_t e = cudaFuncSetAttribute(decode_simt_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(max_ranges, kHeads / kSimtHeads);
  decode_simt_kernel<<<grid, kSimtThreads, smem, stream>>>(
      (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)cache, num_blocks, block_size, block_table,
      max_blocks_per_seq, batch, softmax_scale * 1.4426950408889634f, (__nv_bfloat16 *)out, lse,
      ws, max_ranges, dev_status);
  return cudaGetLastError();
}

}  // namespace mla
