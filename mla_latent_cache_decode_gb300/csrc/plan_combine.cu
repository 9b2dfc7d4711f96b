// Split-KV planner and log-sum-exp combine kernels.
//
// The planner turns the (device-resident) sequence lengths into the plan
// described in common.cuh; the combine kernels merge the fp32 partials of
// requests that were spread over several workers.  Merging partial softmax
// results by their log-sum-exp is standard flash-decoding, used here so that
// one long request does not stall the batch [dp-attention-expert-parallel-mla-
// kv-replication (inferenceinterviews.com), "What it costs"].
#include "common.cuh"

namespace mla {

constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const int32_t *__restrict__ seq_lens,
                                                            int32_t batch, int32_t unit_tokens,
                                                            int32_t max_blocks_per_seq,
                                                            int32_t block_size, int32_t max_ranges,
                                                            void *ws, int32_t heads,
                                                            int32_t *dev_status) {
  PlanView v = plan_view(ws, batch, heads, max_ranges);
  int32_t *seq_out = const_cast<int32_t *>(v.seq_len);
  int32_t *prefix = const_cast<int32_t *>(v.unit_prefix);
  int32_t *range_first = const_cast<int32_t *>(v.range_first);
  __shared__ int32_t warp_sums[kPlanThreads / 32];
  __shared__ int32_t carry;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int64_t max_len = (int64_t)max_blocks_per_seq * block_size;
  if (tid == 0) carry = 0;
  __syncthreads();
  // exclusive scan of units per request, in chunks of kPlanThreads
  for (int base = 0; base < batch; base += kPlanThreads) {
    const int b = base + tid;
    int32_t units = 0;
    if (b < batch) {
      int32_t L = seq_lens[b];
      if (L < 0 || (int64_t)L > max_len) {
        report(dev_status, MLA_ERR_DEVICE_RANGE);
        L = L < 0 ? 0 : (int32_t)max_len;
      }
      seq_out[b] = L;
      units = (L + unit_tokens - 1) / unit_tokens;
      v.counters[2 * b] = 0;
      v.counters[2 * b + 1] = 0;
    }
    int32_t x = units;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int32_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[wid] = x;
    __syncthreads();
    if (wid == 0) {
      int32_t s = warp_sums[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int32_t y = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += y;
      }
      warp_sums[lane] = s;  // inclusive over warps
    }
    __syncthreads();
    const int32_t incl = x + (wid > 0 ? warp_sums[wid - 1] : 0) + carry;
    if (b < batch) prefix[b] = incl - units;
    __syncthreads();
    if (tid == kPlanThreads - 1) carry = incl;
    __syncthreads();
  }
  const int32_t U = carry;
  if (tid == 0) prefix[batch] = U;
  const int32_t P = U < max_ranges ? U : max_ranges;
  __syncthreads();
  // first request of every range: the largest b with prefix[b] <= R_p
  for (int p = tid; p < P; p += kPlanThreads) {
    const int32_t r = range_begin(p, U, P);
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= r) lo = mid; else hi = mid - 1;
    }
    range_first[p] = lo;
  }
  if (tid == 0) {
    PlanHeader *h = const_cast<PlanHeader *>(v.hdr);
    h->total_units = U;
    h->num_ranges = P;
    h->max_ranges = max_ranges;
    h->batch = batch;
    h->unit_tokens = unit_tokens;
    h->max_blocks_per_seq = max_blocks_per_seq;
    h->block_size = block_size;
    h->pad = 0;
  }
}

cudaError_t launch_plan(const int32_t *seq_lens, int32_t batch, int32_t unit_tokens,
                        int32_t max_blocks_per_seq, int32_t block_size, int32_t max_ranges,
                        void *ws, int32_t heads, int32_t *dev_status, cudaStream_t stream) {
  plan_kernel<<<1, kPlanThreads, 0, stream>>>(seq_lens, batch, unit_tokens, max_blocks_per_seq,
                                              block_size, max_ranges, ws, heads, dev_status);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Combine: one warp per (request, head); lane k owns output dims 4k..4k+3 of
// every 128-dim quarter.
// ---------------------------------------------------------------------------
template <typename SlotFn>
__device__ __forceinline__ void combine_head(const float *__restrict__ o_part,
                                             const float *__restrict__ lse_part, int nsplit,
                                             SlotFn slot, int h, int heads,
                                             __nv_bfloat16 *__restrict__ out_row,
                                             float *lse_out) {
  const int lane = threadIdx.x & 31;
  float m = -INFINITY;
  for (int s = lane; s < nsplit; s += 32) m = fmaxf(m, lse_part[(int64_t)slot(s) * heads + h]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float4 acc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  float z = 0.f;
  if (m != -INFINITY) {
    for (int s = 0; s < nsplit; ++s) {
      const int64_t w = slot(s);
      const float l = lse_part[w * heads + h];
      if (l == -INFINITY) continue;
      const float a = __expf(l - m);
      z += a;
      const float4 *src = (const float4 *)(o_part + (w * heads + h) * kVDim);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 x = src[lane + 32 * k];
        acc[k].x += a * x.x; acc[k].y += a * x.y; acc[k].z += a * x.z; acc[k].w += a * x.w;
      }
    }
  }
  const float inv = z > 0.f ? 1.f / z : 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc[k].x * inv, acc[k].y * inv);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc[k].z * inv, acc[k].w * inv);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t *>(&lo);
    pk.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(out_row + 4 * (lane + 32 * k)) = pk;
  }
  if (lse_out && lane == 0) *lse_out = z > 0.f ? m + logf(z) : -INFINITY;
}

// Merges the partials of every split request of a plan.
__global__ void __launch_bounds__(128) plan_combine_kernel(void *ws, int32_t batch, int32_t heads,
                                                           int32_t max_ranges,
                                                           __nv_bfloat16 *__restrict__ out,
                                                           float *__restrict__ lse) {
  PlanView v = plan_view(ws, batch, heads, max_ranges);
  const int b = blockIdx.x;
  const int h = blockIdx.y * 4 + (threadIdx.x >> 5);
  if (h >= heads) return;
  const int32_t U = v.hdr->total_units, P = v.hdr->num_ranges;
  const int32_t Ub = v.unit_prefix[b], n = v.unit_prefix[b + 1] - Ub;
  if (n == 0) return;
  const int32_t p0 = range_of(Ub, U, P), p1 = range_of(Ub + n - 1, U, P);
  if (p0 == p1) return;
  auto slot = [&](int s) { return partial_slot(p0 + s, U, P, Ub); };
  combine_head(v.o_part, v.lse_part, p1 - p0 + 1, slot, h, heads,
               out + ((int64_t)b * heads + h) * kVDim, lse ? lse + (int64_t)b * heads + h : nullptr);
}

cudaError_t launch_plan_combine(void *ws, int32_t batch, int32_t heads, int32_t max_ranges,
                                void *out, float *lse, cudaStream_t stream) {
  dim3 grid(batch, (heads + 3) / 4);
  plan_combine_kernel<<<grid, 128, 0, stream>>>(ws, batch, heads, max_ranges,
                                                (__nv_bfloat16 *)out, lse);
  return cudaGetLastError();
}

// The public combine over caller-given split offsets.
__global__ void __launch_bounds__(128) offsets_combine_kernel(const float *__restrict__ o_part,
                                                              const float *__restrict__ lse_part,
                                                              const int32_t *__restrict__ offsets,
                                                              int32_t heads,
                                                              __nv_bfloat16 *__restrict__ out,
                                                              float *__restrict__ lse) {
  const int b = blockIdx.x;
  const int h = blockIdx.y * 4 + (threadIdx.x >> 5);
  if (h >= heads) return;
  const int32_t w0 = offsets[b], w1 = offsets[b + 1];
  auto slot = [&](int s) { return w0 + s; };
  combine_head(o_part, lse_part, w1 > w0 ? w1 - w0 : 0, slot, h, heads,
               out + ((int64_t)b * heads + h) * kVDim, lse ? lse + (int64_t)b * heads + h : nullptr);
}

cudaError_t launch_offsets_combine(const float *o_part, const float *lse_part,
                                   const int32_t *offsets, int32_t batch, int32_t heads, void *out,
                                   float *lse, cudaStream_t stream) {
  dim3 grid(batch, (heads + 3) / 4);
  offsets_combine_kernel<<<grid, 128, 0, stream>>>(o_part, lse_part, offsets, heads,
                                                   (__nv_bfloat16 *)out, lse);
  return cudaGetLastError();
}

}  // namespace mla
