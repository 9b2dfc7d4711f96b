// mla_cache_append kernel: store each new token's 576-wide latent row
// (the kv_a_proj_with_mqa output, 512 kv_c + 64 k_rope) into its paged slot,
// bit-exactly, as 72 16-byte words per row.
#include "common.cuh"
#include "fp8.cuh"

namespace mla {

constexpr int kWordsPerRow = kRow * 2 / 16;  // 72

__global__ void __launch_bounds__(256) cache_append_kernel(const uint4 *__restrict__ kv_new,
                                                           const int64_t *__restrict__ slots,
                                                           int64_t num_tokens,
                                                           uint4 *__restrict__ cache,
                                                           int64_t num_slots,
                                                           int32_t *dev_status) {
  const int64_t total = num_tokens * kWordsPerRow;
  for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < total;
       k += (int64_t)gridDim.x * blockDim.x) {
    const int64_t tok = k / kWordsPerRow;
    const int word = (int)(k - tok * kWordsPerRow);
    const int64_t slot = __ldg(slots + tok);
    if (slot < 0 || slot >= num_slots) {
      if (slot != -1 && word == 0) report(dev_status, MLA_ERR_DEVICE_RANGE);
      continue;
    }
    cache[slot * kWordsPerRow + word] = __ldg(kv_new + tok * kWordsPerRow + word);
  }
}

cudaError_t launch_cache_append(const void *kv_new, const int64_t *slots, int64_t num_tokens,
                                void *cache, int64_t num_slots, int32_t *dev_status,
                                cudaStream_t stream) {
  const int64_t total = num_tokens * kWordsPerRow;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  cache_append_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
      (const uint4 *)kv_new, slots, num_tokens, (uint4 *)cache, num_slots, dev_status);
  return cudaGetLastError();
}

// FP8 cache: each new bf16 row element x is stored as the E4M3 code nearest
// to fp32(x) * inv_scale (ties to even, saturating to +-448), 576 bytes per
// row, as 72 8-byte words (one per thread: 8 elements from one 16-byte bf16
// word).
__global__ void __launch_bounds__(256) cache_append_fp8_kernel(const uint4 *__restrict__ kv_new,
                                                               const int64_t *__restrict__ slots,
                                                               int64_t num_tokens,
                                                               uint2 *__restrict__ cache,
                                                               int64_t num_slots, float inv_scale,
                                                               int32_t *dev_status) {
  const int64_t total = num_tokens * kWordsPerRow;
  for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < total;
       k += (int64_t)gridDim.x * blockDim.x) {
    const int64_t tok = k / kWordsPerRow;
    const int word = (int)(k - tok * kWordsPerRow);
    const int64_t slot = __ldg(slots + tok);
    if (slot < 0 || slot >= num_slots) {
      if (slot != -1 && word == 0) report(dev_status, MLA_ERR_DEVICE_RANGE);
      continue;
    }
    cache[slot * kWordsPerRow + word] = quantize_bf16x8(__ldg(kv_new + tok * kWordsPerRow + word),
                                                        inv_scale);
  }
}

cudaError_t launch_cache_append_fp8(const void *kv_new, const int64_t *slots, int64_t num_tokens,
                                    void *cache, int64_t num_slots, float inv_scale,
                                    int32_t *dev_status, cudaStream_t stream) {
  const int64_t total = num_tokens * kWordsPerRow;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  cache_append_fp8_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
      (const uint4 *)kv_new, slots, num_tokens, (uint2 *)cache, num_slots, inv_scale, dev_status);
  return cudaGetLastError();
}

}  // namespace mla
