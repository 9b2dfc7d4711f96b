// Log-sum-exp merge of split partials for the combine kernels: partial w
// of request b holds its own normalised output o_w (bf16) and lse_w (fp32),
// and out = sum_w e^(lse_w - M) o_w / sum_w e^(lse_w - M), lse = M + log sum,
// M = max_w lse_w, accumulated in fp32 (standard split-KV decoding; it keeps
// one long request from stalling the batch [dp-attention-expert-parallel-
// mla-kv-replication (inferenceinterviews.com), "What it costs"]).
#pragma once

#include "common.cuh"

namespace mla {

constexpr int kCombDims = 16;   // output dims of one merge item (one thread per head)
constexpr int kCombGroup = 4;   // splits per lane whose loads are in flight together

// Slot of the k-th split of a request (see ReqSplit).
__device__ __forceinline__ int64_t split_slot(const ReqSplit &rs, int k) {
  return k == 0 ? 2 * rs.p0 + rs.first_odd : 2 * (rs.p0 + k);
}

// A split record that stays within the partial slots: a plan made for other
// arguments (which the decode reports) may hold anything.
__device__ __forceinline__ bool split_in_bounds(const ReqSplit &rs, int32_t max_ranges) {
  return rs.p0 >= 0 && rs.p0 <= rs.p1 && rs.p1 < max_ranges;
}

// Lane sl of kLanes merges splits sl, sl + kLanes, ... of request rs for
// head h and output dims [d0, d0 + 16), kCombGroup at a time with their loads
// in flight before any is used (a warp's 16-byte loads are 512 contiguous
// bytes of 32 heads); the running max rescales what was summed so far.
// Partials are bf16 [slot][512 / 8][128][8], lse fp32 [slot][128].
template <int kLanes>
__device__ __forceinline__ void accumulate_splits(const PlanView &v, const ReqSplit &rs, int sl,
                                                  int h, int d0, float4 (&acc)[kCombDims / 4],
                                                  float &m, float &z) {
  const int nsplit = rs.p1 - rs.p0 + 1;
#pragma unroll
  for (int j = 0; j < kCombDims / 4; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  m = -INFINITY;
  z = 0.f;
  for (int k0 = sl; k0 < nsplit; k0 += kLanes * kCombGroup) {
    float l[kCombGroup];
    float4 x[kCombGroup][kCombDims / 4];
#pragma unroll
    for (int u = 0; u < kCombGroup; ++u) {
      const int k = k0 + u * kLanes;
      const int64_t w = split_slot(rs, k < nsplit ? k : k0);  // k0 < nsplit: a valid slot
      l[u] = k < nsplit ? v.lse_part[w * kHeads + h] : -INFINITY;
      const uint4 *src = reinterpret_cast<const uint4 *>(v.o_part) +
                         (w * (kVDim / 8) + d0 / 8) * kHeads + h;
#pragma unroll
      for (int j = 0; j < kCombDims / 8; ++j) {
        const uint4 raw = __ldg(src + (int64_t)j * kHeads);
        x[u][2 * j] = make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xffff0000u),
                                  __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xffff0000u));
        x[u][2 * j + 1] = make_float4(__uint_as_float(raw.z << 16), __uint_as_float(raw.z & 0xffff0000u),
                                      __uint_as_float(raw.w << 16), __uint_as_float(raw.w & 0xffff0000u));
      }
    }
    float mc = m;
#pragma unroll
    for (int u = 0; u < kCombGroup; ++u) mc = fmaxf(mc, l[u]);
    if (mc == -INFINITY) continue;
    if (m != -INFINITY && mc != m) {
      const float r = __expf(m - mc);
      z *= r;
#pragma unroll
      for (int j = 0; j < kCombDims / 4; ++j) {
        acc[j].x *= r; acc[j].y *= r; acc[j].z *= r; acc[j].w *= r;
      }
    }
    m = mc;
#pragma unroll
    for (int u = 0; u < kCombGroup; ++u) {
      const float a = l[u] == -INFINITY ? 0.f : __expf(l[u] - m);
      z += a;
#pragma unroll
      for (int j = 0; j < kCombDims / 4; ++j) {
        acc[j].x += a * x[u][j].x; acc[j].y += a * x[u][j].y;
        acc[j].z += a * x[u][j].z; acc[j].w += a * x[u][j].w;
      }
    }
  }
}

// One lane's finished merge (kLanes = 1) into a row of the bf16 staging tile;
// returns the head's lse.
__device__ __forceinline__ float finish_row16(const float4 (&acc)[kCombDims / 4], float m, float z,
                                              __nv_bfloat16 *tile_row) {
  const float inv = z > 0.f ? 1.f / z : 0.f;
#pragma unroll
  for (int j = 0; j < kCombDims / 4; ++j) {
    *reinterpret_cast<__nv_bfloat162 *>(tile_row + 4 * j) =
        __floats2bfloat162_rn(acc[j].x * inv, acc[j].y * inv);
    *reinterpret_cast<__nv_bfloat162 *>(tile_row + 4 * j + 2) =
        __floats2bfloat162_rn(acc[j].z * inv, acc[j].w * inv);
  }
  return z > 0.f ? m + logf(z) : -INFINITY;
}

}  // namespace mla
