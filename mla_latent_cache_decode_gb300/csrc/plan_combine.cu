// Split-KV planner and log-sum-exp combine kernels.
//
// The planner turns the (device-resident) sequence lengths into the plan
// described in common.cuh; the combine kernels merge, in fp32, the partials
// (bf16 outputs with fp32 log-sum-exps; fp32 for the public mla_combine) of
// requests that were spread over several workers.  Merging partial softmax
// results by their log-sum-exp is standard flash-decoding, used here so that
// one long request does not stall the batch [dp-attention-expert-parallel-mla-
// kv-replication (inferenceinterviews.com), "What it costs"].
#include "common.cuh"
#include "merge.cuh"
#include "sm100.cuh"

namespace mla {

// The planner is one block whose phases are short dependent chains between
// barriers; every warp issues every phase, so it runs 8 warps (2 per SM
// sub-partition) rather than 32 and loops where a batch or the ranges exceed
// a pass.
constexpr int kPlanThreads = 256;
constexpr int kPlanWarps = kPlanThreads / 32;
constexpr int kMaxPlanRanges = 1024;  // boundaries are settled in shared memory
constexpr int kPlanChunks = (kMaxPlanRanges + 1 + 31) / 32;  // 32-boundary chunks
// Batches up to this size keep their prefixes and lengths in shared memory
// too, so the planner's binary searches and walks make no global round trips
// (larger batches read them back from the workspace).
constexpr int kPlanSmemBatch = 2048;

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const int32_t *__restrict__ seq_lens,
                                                            const int32_t *__restrict__ block_table,
                                                            int64_t num_blocks,
                                                            int32_t batch, int32_t unit_tokens,
                                                            int32_t max_blocks_per_seq,
                                                            int32_t block_size, int32_t max_ranges,
                                                            void *ws, int32_t heads,
                                                            int32_t *dev_status) {
  PlanView v = plan_view(ws, batch, heads, max_ranges);
  int32_t *seq_out = const_cast<int32_t *>(v.seq_len);
  int32_t *prefix = const_cast<int32_t *>(v.unit_prefix);
  int32_t *range_start = const_cast<int32_t *>(v.range_start);
  int32_t *range_first = const_cast<int32_t *>(v.range_first);
  int64_t *cost_prefix = const_cast<int64_t *>(v.cost_prefix);
  __shared__ int64_t warp_sums[kPlanWarps];
  __shared__ int64_t carry;
  __shared__ int32_t chunk_ext[kPlanChunks];
  __shared__ int32_t bound[kMaxPlanRanges + 1];
  __shared__ int32_t s_rfirst[kMaxPlanRanges];
  __shared__ int32_t s_prefix[kPlanSmemBatch + 1], s_seq[kPlanSmemBatch];
  __shared__ int64_t s_cost[kPlanSmemBatch + 1];
  const bool small = batch <= kPlanSmemBatch;
  // where the phases below read the prefixes and clamped lengths back from
  const int32_t *pre = small ? s_prefix : prefix;
  const int64_t *cpre = small ? s_cost : cost_prefix;
  const int32_t *sq = small ? s_seq : seq_out;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int64_t max_len = (int64_t)max_blocks_per_seq * block_size;
  if (tid == 0) carry = 0;
  __syncthreads();
  // Exclusive scan of (non-empty requests, units) per request, packed in one
  // int64 (count in the high word, units in the low; the host bounds the
  // total units below 2^31, so the low word never carries).
  for (int base = 0; base < batch; base += kPlanThreads) {
    const int b = base + tid;
    int64_t item = 0;
    if (b < batch) {
      int32_t L = seq_lens[b];
      if (L < 0 || (int64_t)L > max_len) {
        report(dev_status, MLA_ERR_DEVICE_RANGE);
        L = L < 0 ? 0 : (int32_t)max_len;
      }
      seq_out[b] = L;
      if (small) s_seq[b] = L;
      const int32_t units = (L + unit_tokens - 1) / unit_tokens;
      item = units > 0 ? (int64_t(1) << 32) | units : 0;
      v.counters[2 * b] = 0;
      v.counters[2 * b + 1] = 0;
    }
    int64_t x = item;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[wid] = x;
    __syncthreads();
    if (wid == 0) {
      int64_t s = lane < kPlanWarps ? warp_sums[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += y;
      }
      if (lane < kPlanWarps) warp_sums[lane] = s;  // inclusive over warps
    }
    __syncthreads();
    const int64_t incl = x + (wid > 0 ? warp_sums[wid - 1] : 0) + carry;
    if (b < batch) {
      const int64_t excl = incl - item;
      const int32_t pb = (int32_t)(excl & 0xffffffff);
      const int64_t cb = kUnitCost * (excl & 0xffffffff) + kSegmentCost * (excl >> 32);
      prefix[b] = pb;
      cost_prefix[b] = cb;
      if (small) {
        s_prefix[b] = pb;
        s_cost[b] = cb;
      }
    }
    __syncthreads();
    if (tid == kPlanThreads - 1) carry = incl;
    __syncthreads();
  }
  const int32_t U = (int32_t)(carry & 0xffffffff);
  const int64_t C = kUnitCost * U + kSegmentCost * (carry >> 32);
  if (tid == 0) {
    prefix[batch] = U;
    cost_prefix[batch] = C;
    if (small) {
      s_prefix[batch] = U;
      s_cost[batch] = C;
    }
  }
  __syncthreads();  // the shared copies are complete
  const int32_t P = U < max_ranges ? U : max_ranges;
  // Range boundaries.  First the unit at cost p*C/P, held as R_p - p ...
  for (int p = tid; p <= P; p += kPlanThreads) {
    int32_t r = 0;
    if (p == P) {
      r = U;
    } else if (p > 0) {
      const int64_t c = (int64_t)p * C / P;
      int lo = 0, hi = batch - 1;  // the request whose cost span holds c
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cpre[mid] <= c) lo = mid; else hi = mid - 1;
      }
      const int64_t x = c - cpre[lo];
      const int64_t k = x < kSegmentCost ? 0 : (x - kSegmentCost + kUnitCost / 2) / kUnitCost;
      const int32_t n = pre[lo + 1] - pre[lo];
      r = pre[lo] + (int32_t)(k < n ? k : n);
    }
    bound[p] = r - p;
  }
  __syncthreads();
  // ... then the least change that makes them strictly increasing with
  // R_0 = 0 and R_P = U: R_p = p + min over q >= p of (max over q' <= q of
  // (R_q' - q')), the last term pinned to U - P.  R_0 = 0 and R_P = U hold
  // already; when every range also got a unit (R_p - p non-decreasing, the
  // usual case) the scans would change nothing.  Otherwise both run over
  // chunks of 32 boundaries, one chunk a warp, and then take the other
  // chunks' extremes in.
  bool rising = true;
  for (int p = tid; p < P; p += kPlanThreads) rising = rising && bound[p] <= bound[p + 1];
  const bool fix = !__syncthreads_and(rising);
  const int nch = (P + 1 + 31) / 32;
  if (!fix) {
    for (int p = tid; p <= P; p += kPlanThreads) bound[p] += p;
  } else if (P > 0) {
    for (int ch = wid; ch < nch; ch += kPlanWarps) {  // prefix max within chunks
      const int p = ch * 32 + lane;
      int32_t x = p <= P ? bound[p] : INT32_MIN;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x = max(x, y);
      }
      if (p <= P) bound[p] = x;
      if (lane == 31) chunk_ext[ch] = x;
    }
    __syncthreads();
    for (int ch = wid; ch < nch; ch += kPlanWarps) {  // ... and over the chunks before
      int32_t c = INT32_MIN;
      for (int k = lane; k < ch; k += 32) c = max(c, chunk_ext[k]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) c = max(c, __shfl_xor_sync(0xffffffffu, c, o));
      const int p = ch * 32 + lane;
      if (p <= P) bound[p] = p == P ? U - P : max(bound[p], c);
    }
    __syncthreads();
    for (int ch = wid; ch < nch; ch += kPlanWarps) {  // suffix min within chunks (from the top)
      const int p = P - (ch * 32 + lane);
      int32_t x = p >= 0 ? bound[p] : INT32_MAX;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x = min(x, y);
      }
      if (p >= 0) bound[p] = x;
      if (lane == 31) chunk_ext[ch] = x;
    }
    __syncthreads();
    for (int ch = wid; ch < nch; ch += kPlanWarps) {  // ... and over the chunks above
      int32_t c = INT32_MAX;
      for (int k = lane; k < ch; k += 32) c = min(c, chunk_ext[k]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) c = min(c, __shfl_xor_sync(0xffffffffu, c, o));
      const int p = P - (ch * 32 + lane);
      if (p >= 0) bound[p] = min(bound[p], c) + p;
    }
  }
  __syncthreads();
  for (int p = tid; p <= max_ranges; p += kPlanThreads) range_start[p] = p <= P ? bound[p] : U;
  // first request of every range: the largest b with prefix[b] <= R_p
  for (int p = tid; p < P; p += kPlanThreads) {
    const int32_t r = bound[p];
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= r) lo = mid; else hi = mid - 1;
    }
    range_first[p] = lo;
    s_rfirst[p] = lo;  // read below by this thread only (the same p)
  }
  // every request's split, for the combine (see ReqSplit)
  auto range_of = [&](int32_t u) {  // the largest p < P with R_p <= u
    int lo = 0, hi = P - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (bound[mid] <= u) lo = mid; else hi = mid - 1;
    }
    return lo;
  };
  // (requests from the block's last thread down, so that a small batch's
  // splits and the ranges' records below go to different warps)
  ReqSplit *req_split = const_cast<ReqSplit *>(v.req_split);
  for (int b = kPlanThreads - 1 - tid; b < batch; b += kPlanThreads) {
    const int32_t Ub = pre[b], n = pre[b + 1] - Ub;
    ReqSplit r;
    r.p0 = n > 0 ? range_of(Ub) : 0;
    r.p1 = n > 0 ? range_of(Ub + n - 1) : 0;
    r.first_odd = n > 0 && bound[r.p0] < Ub ? 1 : 0;
    r.pad = 0;
    req_split[b] = r;
  }
  // the first kSegCache segments of every range (see SegRec)
  int32_t *seg_count = const_cast<int32_t *>(v.seg_count);
  SegRec *seg_rec = const_cast<SegRec *>(v.seg_rec);
  const int32_t stamp =
      plan_stamp(batch, max_ranges, unit_tokens, block_size, max_blocks_per_seq);
  const bool rows = block_table && block_size >= unit_tokens;
  for (int p = tid; p < max_ranges; p += kPlanThreads) {
    int32_t n = 0;
    if (p < P) {
      const int32_t r0 = bound[p], r1 = bound[p + 1];
      // the first kSegCache segments, their table entries loaded together
      int b = s_rfirst[p];
      SegRec rec[kSegCache];
      int32_t blk[kSegCache];
#pragma unroll
      for (int i = 0; i < kSegCache; ++i) {
        while (b < batch && pre[b] < r1 && pre[b + 1] <= max(r0, pre[b])) ++b;  // empty ones
        blk[i] = -1;
        if (b < batch && pre[b] < r1) {
          const int32_t Ub = pre[b], Ue = pre[b + 1];
          const int32_t u0 = max(r0, Ub), u1 = min(r1, Ue);
          rec[i].b = b;
          rec[i].t0 = (u0 - Ub) * unit_tokens;
          rec[i].t1 = min((u1 - Ub) * unit_tokens, sq[b]);
          rec[i].slot = segment_slot(p, r0, r1, Ub, Ue);
          if (rows && rec[i].t0 < rec[i].t1)
            blk[i] = block_table[(int64_t)b * max_blocks_per_seq + rec[i].t0 / block_size];
          ++n;
          ++b;
        }
      }
#pragma unroll
      for (int i = 0; i < kSegCache; ++i) {
        if (i < n) {
          SegRec r = rec[i];
          r.row0 = blk[i] >= 0 && (int64_t)blk[i] < num_blocks
                       ? blk[i] * block_size + r.t0 % block_size
                       : -1;
          r.stamp = stamp;
          r.pad1 = r.pad2 = 0;
          seg_rec[(int64_t)p * kSegCache + i] = r;
        }
      }
      // the count of the rest
      for (; b < batch && pre[b] < r1; ++b)
        if (min(r1, pre[b + 1]) > max(r0, pre[b])) ++n;
    }
    seg_count[p] = n;
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

cudaError_t launch_plan(const int32_t *seq_lens, const int32_t *block_table, int64_t num_blocks,
                        int32_t batch, int32_t unit_tokens, int32_t max_blocks_per_seq,
                        int32_t block_size, int32_t max_ranges, void *ws, int32_t heads,
                        int32_t *dev_status, cudaStream_t stream) {
  if (max_ranges < 1 || max_ranges > kMaxPlanRanges ||
      !plan_fits(batch, max_blocks_per_seq, block_size, unit_tokens))
    return cudaErrorInvalidValue;
  plan_kernel<<<1, kPlanThreads, 0, stream>>>(seq_lens, block_table, num_blocks, batch,
                                              unit_tokens, max_blocks_per_seq, block_size,
                                              max_ranges, ws, heads, dev_status);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Combine: one block of 128 threads per (request, head) row; thread t owns
// output dims 4t..4t+3.  The partials were just written by the decode and sit
// in L2, so the kernel is latency-bound: many rows in flight and the split
// loop unrolled so that several partial loads are outstanding per thread.
// ---------------------------------------------------------------------------
constexpr int kCombineThreads = kVDim / 4;  // 128

template <typename SlotFn>
__device__ __forceinline__ void combine_row(const float *__restrict__ o_part,
                                            const float *__restrict__ lse_part, int nsplit,
                                            SlotFn slot, int h, int heads,
                                            __nv_bfloat16 *__restrict__ out_row,
                                            float *lse_out) {
  // The block's splits are taken kCombineThreads at a time: thread t works
  // out the slot and log-sum-exp of split base + t once, in shared memory,
  // and every thread of the block reads them from there.
  __shared__ int64_t s_slot[kCombineThreads];
  __shared__ float s_lse[kCombineThreads];
  const int t = threadIdx.x;
  float m = -INFINITY;
  for (int base = 0; base < nsplit; base += kCombineThreads) {
    const int cnt = min(kCombineThreads, nsplit - base);
    __syncthreads();
    if (t < cnt) {
      const int64_t w = slot(base + t);
      s_slot[t] = w;
      s_lse[t] = lse_part[w * heads + h];
    }
    __syncthreads();
    for (int k = 0; k < cnt; ++k) m = fmaxf(m, s_lse[k]);
  }
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float z = 0.f;
  if (m != -INFINITY) {
    for (int base = 0; base < nsplit; base += kCombineThreads) {
      const int cnt = min(kCombineThreads, nsplit - base);
      if (nsplit > kCombineThreads) {  // else the table from the max pass is still in place
        __syncthreads();
        if (t < cnt) {
          const int64_t w = slot(base + t);
          s_slot[t] = w;
          s_lse[t] = lse_part[w * heads + h];
        }
        __syncthreads();
      }
#pragma unroll 4
      for (int k = 0; k < cnt; ++k) {
        const float l = s_lse[k];
        const float a = l == -INFINITY ? 0.f : __expf(l - m);
        const float4 x =
            __ldg(reinterpret_cast<const float4 *>(o_part + (s_slot[k] * heads + h) * kVDim) + t);
        z += a;
        acc.x += a * x.x; acc.y += a * x.y; acc.z += a * x.z; acc.w += a * x.w;
      }
    }
  }
  const float inv = z > 0.f ? 1.f / z : 0.f;
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t *>(&lo);
  pk.y = *reinterpret_cast<uint32_t *>(&hi);
  *reinterpret_cast<uint2 *>(out_row + 4 * t) = pk;
  if (lse_out && t == 0) *lse_out = z > 0.f ? m + logf(z) : -INFINITY;
}

// Merges the partials of every split request of a plan.  The decode stores
// them in bf16 as [slot][512 / 8][128][8].  A block takes one request and 16
// output dims.  With one split lane (kLanes = 1) its thread h is head h and
// merges all the request's splits, four at a time with their loads all in
// flight before any is used (a warp's 16-byte loads are 512 contiguous bytes
// of 32 heads), in fp32.  With kLanes = 4 or 16 split lanes (small batches,
// whose requests are spread over many ranges) a block takes 128 / kLanes
// heads, and lane s (threads s * 128 / kLanes ...) merges splits s, s + kLanes,
// s + 2 kLanes, ... of them; the kLanes running results of a head (max, weight
// sum, 16 weighted dims) are then merged through shared memory, each thread
// finishing 16 / kLanes dims of one head.  The bf16 results leave as 32-byte
// row pieces.  grid = (batch, 512 / 16, kLanes), 128 threads.

template <int kLanes>
__global__ void __launch_bounds__(kHeads) plan_combine_kernel(void *ws, int32_t batch,
                                                              int32_t max_ranges,
                                                              __nv_bfloat16 *__restrict__ out,
                                                              float *__restrict__ lse) {
  constexpr int kBlockHeads = kHeads / kLanes;
  // the next layer's decode may launch its prologue meanwhile (it waits for
  // this grid before it reads or writes anything this one touches)
  sm100::griddep_launch_dependents();
  // launched as a programmatic dependent of the decode, this block may start
  // before the decode ends: the partials are read only once it has completed
  sm100::griddep_wait();
  PlanView v = plan_view(ws, batch, kHeads, max_ranges);
  const int b = blockIdx.x, d0 = blockIdx.y * kCombDims;
  const int sl = (int)threadIdx.x / kBlockHeads;  // split lane
  const int hb = (int)threadIdx.x % kBlockHeads;  // head in the block
  const int h = blockIdx.z * kBlockHeads + hb;
  const ReqSplit rs = v.req_split[b];
  if (rs.p0 == rs.p1) return;  // not split (or empty): the decode wrote it
  if (!split_in_bounds(rs, max_ranges)) return;
  __shared__ __align__(16) __nv_bfloat16 tile[kBlockHeads][kCombDims + 8];  // +8: stagger
  float4 acc[kCombDims / 4];
  float m, z;
  accumulate_splits<kLanes>(v, rs, sl, h, d0, acc, m, z);
  if constexpr (kLanes == 1) {
    const float lse_h = finish_row16(acc, m, z, &tile[hb][0]);
    if (lse && blockIdx.y == 0) lse[(int64_t)b * kHeads + h] = lse_h;
  } else {
    constexpr int kDimsPerThread = kCombDims / kLanes;
    __shared__ float s_m[kLanes][kBlockHeads], s_z[kLanes][kBlockHeads];
    __shared__ float s_acc[kLanes][kCombDims][kBlockHeads];
    s_m[sl][hb] = m;
    s_z[sl][hb] = z;
#pragma unroll
    for (int j = 0; j < kCombDims / 4; ++j) {
      s_acc[sl][4 * j][hb] = acc[j].x;
      s_acc[sl][4 * j + 1][hb] = acc[j].y;
      s_acc[sl][4 * j + 2][hb] = acc[j].z;
      s_acc[sl][4 * j + 3][hb] = acc[j].w;
    }
    __syncthreads();
    // thread (sl, hb) finishes dims [sl kDimsPerThread, (sl + 1) kDimsPerThread) of head hb
    float M = -INFINITY;
#pragma unroll
    for (int i = 0; i < kLanes; ++i) M = fmaxf(M, s_m[i][hb]);
    float Z = 0.f;
    float o[kDimsPerThread];
#pragma unroll
    for (int j = 0; j < kDimsPerThread; ++j) o[j] = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int i = 0; i < kLanes; ++i) {
        const float mi = s_m[i][hb];
        const float a = mi == -INFINITY ? 0.f : __expf(mi - M);
        Z += a * s_z[i][hb];
#pragma unroll
        for (int j = 0; j < kDimsPerThread; ++j) o[j] += a * s_acc[i][sl * kDimsPerThread + j][hb];
      }
    }
    const float inv = Z > 0.f ? 1.f / Z : 0.f;
#pragma unroll
    for (int j = 0; j < kDimsPerThread; ++j)
      tile[hb][sl * kDimsPerThread + j] = __float2bfloat16_rn(o[j] * inv);
    if (lse && blockIdx.y == 0 && sl == 0)
      lse[(int64_t)b * kHeads + h] = Z > 0.f ? M + logf(Z) : -INFINITY;
  }
  __syncthreads();
  // kBlockHeads rows x (2 kCombDims) bytes, in 16-byte pieces
  constexpr int kPieces = kCombDims / 8;
  for (int piece = threadIdx.x; piece < kBlockHeads * kPieces; piece += kHeads) {
    const int row = piece / kPieces, part = piece % kPieces;
    __nv_bfloat16 *orow =
        out + ((int64_t)b * kHeads + blockIdx.z * kBlockHeads + row) * kVDim + d0;
    *reinterpret_cast<uint4 *>(orow + part * 8) =
        *reinterpret_cast<const uint4 *>(&tile[row][part * 8]);
  }
}

cudaError_t launch_plan_combine(void *ws, int32_t batch, int32_t heads, int32_t max_ranges,
                                void *out, float *lse, cudaStream_t stream, bool early) {
  if (heads != kHeads) return cudaErrorInvalidValue;
  // Split lanes when requests average four or more ranges (a small batch,
  // where one long request may be spread over most of the SM pairs): 16 from
  // eight ranges a request on average, 4 from four; one otherwise, so that an
  // ordinary batch keeps one block per 16 dims.
  const int lanes =
      (int64_t)batch * 8 <= max_ranges ? 16 : ((int64_t)batch * 4 <= max_ranges ? 4 : 1);
  // early: a programmatic dependent of the decode, whose CTAs release it once
  // they have requested their last tile
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(batch, kVDim / kCombDims, lanes);
  cfg.blockDim = dim3(kHeads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = early ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  __nv_bfloat16 *o = (__nv_bfloat16 *)out;
  if (lanes == 16)
    return cudaLaunchKernelEx(&cfg, plan_combine_kernel<16>, ws, batch, max_ranges, o, lse);
  if (lanes == 4)
    return cudaLaunchKernelEx(&cfg, plan_combine_kernel<4>, ws, batch, max_ranges, o, lse);
  return cudaLaunchKernelEx(&cfg, plan_combine_kernel<1>, ws, batch, max_ranges, o, lse);
}

// Merges the partials of the few-head kernel (decode_tp.cu), stored in bf16
// as [slot][head][512] with fp32 log-sum-exps [slot][head].  A block of 64
// threads takes one (request, head); thread t merges dims [8 t, 8 t + 8) over
// all the request's splits, four at a time with their loads in flight, in
// fp32.  grid = (batch, heads).
constexpr int kTpCombThreads = kVDim / 8;  // 64

__global__ void __launch_bounds__(kTpCombThreads) tp_combine_kernel(void *ws, int32_t batch,
                                                                    int32_t heads,
                                                                    int32_t max_ranges,
                                                                    __nv_bfloat16 *__restrict__ out,
                                                                    float *__restrict__ lse) {
  PlanView v = plan_view(ws, batch, heads, max_ranges);
  const int b = blockIdx.x, h = blockIdx.y, t = threadIdx.x;
  const ReqSplit rs = v.req_split[b];
  if (rs.p0 == rs.p1) return;  // not split (or empty): the decode wrote it
  // a plan made for other arguments (the decode reports it): stay inside the
  // partials' slots whatever the record holds
  if (rs.p0 < 0 || rs.p0 > rs.p1 || rs.p1 >= max_ranges) return;
  const int nsplit = rs.p1 - rs.p0 + 1;
  auto slot_of_split = [&](int k) -> int64_t {
    return k == 0 ? 2 * rs.p0 + rs.first_odd : 2 * (rs.p0 + k);
  };
  float m = -INFINITY;
  for (int k = 0; k < nsplit; ++k) m = fmaxf(m, v.lse_part[slot_of_split(k) * heads + h]);
  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.f;
  float z = 0.f;
  if (m != -INFINITY) {
    for (int k0 = 0; k0 < nsplit; k0 += kCombGroup) {
      float l[kCombGroup];
      uint4 raw[kCombGroup];
#pragma unroll
      for (int u = 0; u < kCombGroup; ++u) {
        const int k = k0 + u;
        const int64_t w = slot_of_split(k < nsplit ? k : k0);
        l[u] = k < nsplit ? v.lse_part[w * heads + h] : -INFINITY;
        raw[u] = __ldg(reinterpret_cast<const uint4 *>(v.o_part + (w * heads + h) * kVDim) + t);
      }
#pragma unroll
      for (int u = 0; u < kCombGroup; ++u) {
        const float a = l[u] == -INFINITY ? 0.f : __expf(l[u] - m);
        z += a;
        const uint32_t w4[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[2 * j] += a * __uint_as_float(w4[j] << 16);
          acc[2 * j + 1] += a * __uint_as_float(w4[j] & 0xffff0000u);
        }
      }
    }
  }
  const float inv = z > 0.f ? 1.f / z : 0.f;
  uint4 o;
  uint32_t *ow = reinterpret_cast<uint32_t *>(&o);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    __nv_bfloat162 pr = __floats2bfloat162_rn(acc[2 * j] * inv, acc[2 * j + 1] * inv);
    ow[j] = *reinterpret_cast<uint32_t *>(&pr);
  }
  reinterpret_cast<uint4 *>(out + ((int64_t)b * heads + h) * kVDim)[t] = o;
  if (lse && t == 0) lse[(int64_t)b * heads + h] = z > 0.f ? m + logf(z) : -INFINITY;
}

cudaError_t launch_tp_combine(void *ws, int32_t batch, int32_t heads, int32_t max_ranges,
                              void *out, float *lse, cudaStream_t stream) {
  if (heads < 1 || heads > 65535) return cudaErrorInvalidValue;
  dim3 grid(batch, heads);
  tp_combine_kernel<<<grid, kTpCombThreads, 0, stream>>>(ws, batch, heads, max_ranges,
                                                         (__nv_bfloat16 *)out, lse);
  return cudaGetLastError();
}

// The public combine over caller-given split offsets.  grid = (batch, heads).
__global__ void __launch_bounds__(kCombineThreads) offsets_combine_kernel(
    const float *__restrict__ o_part, const float *__restrict__ lse_part,
    const int32_t *__restrict__ offsets, int32_t heads, __nv_bfloat16 *__restrict__ out,
    float *__restrict__ lse) {
  const int b = blockIdx.x, h = blockIdx.y;
  const int32_t w0 = offsets[b], w1 = offsets[b + 1];
  auto slot = [&](int s) { return w0 + s; };
  combine_row(o_part, lse_part, w1 > w0 ? w1 - w0 : 0, slot, h, heads,
              out + ((int64_t)b * heads + h) * kVDim, lse ? lse + (int64_t)b * heads + h : nullptr);
}

cudaError_t launch_offsets_combine(const float *o_part, const float *lse_part,
                                   const int32_t *offsets, int32_t batch, int32_t heads, void *out,
                                   float *lse, cudaStream_t stream) {
  dim3 grid(batch, heads);
  offsets_combine_kernel<<<grid, kCombineThreads, 0, stream>>>(o_part, lse_part, offsets, heads,
                                                               (__nv_bfloat16 *)out, lse);
  return cudaGetLastError();
}

}  // namespace mla
