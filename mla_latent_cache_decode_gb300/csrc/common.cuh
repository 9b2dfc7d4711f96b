// Shared device-side definitions for libmla: sizes, status reporting, the
// split-KV plan layout in the workspace.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mla.h"

namespace mla {

constexpr int kRow = MLA_ROW_DIM;        // 576: 512 kv_c + 64 k_rope
constexpr int kVDim = MLA_KV_LORA_RANK;  // 512
constexpr int kHeads = MLA_NUM_HEADS;    // 128

// First error wins; the kernels never trap.
__device__ __forceinline__ void report(int32_t *dev_status, int32_t code) {
  if (dev_status) atomicCAS(dev_status, 0, code);
}

// ---------------------------------------------------------------------------
// Split-KV plan.
//
// Every request b is cut into units of kUnit tokens; unit u of the flattened
// sequence (requests in order) is U_b + i for the i-th unit of request b.
// The U units are split into P = min(P_max, U) contiguous, non-empty ranges,
// range p = [R_p, R_{p+1}), R_0 = 0, R_P = U, stored in range_start.  Range p
// is processed by one worker (a CTA pair for the tensor-core kernel).  The
// boundaries balance cost rather than units: a range costs kUnitCost per unit
// plus kSegmentCost for every request that starts inside it, since each
// segment after a worker's first stages a new query, writes the previous
// segment's result and refills the pipeline.  R_p is the unit at cost
// p * C / P along the batch (C the total cost, each request's start cost
// placed before its units; a target inside a start cost snaps to the
// request's first unit), then moved the least needed to keep every range
// non-empty.  A request whose units lie in one range is written directly; a
// request spanning k ranges leaves k partials (bf16 outputs with fp32
// log-sum-exps) which are merged by log-sum-exp in fp32.  Range p holds at most two partial segments (its first and its
// last), stored in slots 2p and 2p+1: the segment of request b in range p
// uses slot 2p if R_p >= U_b (the range starts inside or at b) and 2p+1
// otherwise.
// ---------------------------------------------------------------------------
constexpr int64_t kUnitCost = 2;
constexpr int64_t kSegmentCost = 7;  // 3.5 units: a segment switch, measured

// Units are counted in int32: the longest batch the table allows must fit.
inline bool plan_fits(int32_t batch, int32_t max_blocks_per_seq, int32_t block_size,
                      int32_t unit_tokens) {
  const int64_t max_len = (int64_t)max_blocks_per_seq * block_size;
  return max_len <= (int64_t)INT32_MAX / 2 &&
         (int64_t)batch * ((max_len + unit_tokens - 1) / unit_tokens) <= (int64_t)INT32_MAX;
}

// Partial slot of the segment of request b (units [Ub, Ue)) in range p =
// [r0, r1), -1 when the request lies wholly in the range.
__host__ __device__ inline int32_t segment_slot(int32_t p, int32_t r0, int32_t r1, int32_t Ub,
                                                int32_t Ue) {
  return Ub < r0 || Ue > r1 ? 2 * p + (r0 < Ub ? 1 : 0) : -1;
}

// The first kSegCache segments of every range, written by the planner so that
// a worker learns its work with one memory round trip: request b, tokens
// [t0, t1), the partial slot (-1: the request is not split, the segment
// writes the output directly), and — when the plan was given the block table
// and pages hold at least a tile — the cache row of the segment's first token
// (row0, -1 if unknown), so its first tile can be loaded without a table
// lookup.  Later segments are found by walking the plan.
constexpr int kSegCache = 4;
struct __align__(16) SegRec {
  int32_t b, t0, t1, slot;
  int32_t row0;
  int32_t stamp;  // plan_stamp of the arguments the plan was made for
  int32_t pad1, pad2;
};

// A 32-bit mix of the arguments a plan is made for.  The planner writes it
// into every segment record and a decode compares it with its own arguments
// on each record it reads (already in registers: no extra load), so a plan
// made for another batch, head count, page size or table width is refused.
__host__ __device__ inline int32_t plan_stamp(int32_t batch, int32_t max_ranges,
                                              int32_t unit_tokens, int32_t block_size,
                                              int32_t max_blocks_per_seq) {
  uint32_t h = 0x6d2b79f5u;
  const uint32_t parts[5] = {(uint32_t)batch, (uint32_t)max_ranges, (uint32_t)unit_tokens,
                             (uint32_t)block_size, (uint32_t)max_blocks_per_seq};
  for (int i = 0; i < 5; ++i) {
    h ^= parts[i] + 0x9e3779b9u + (h << 6) + (h >> 2);
    h *= 0x85ebca6bu;
  }
  return (int32_t)(h ^ (h >> 15));
}

// Split of request b, written by the planner for the combine: its partials
// are in ranges p0..p1 (p0 == p1: not split), stored in slots
// 2 p0 + first_odd, 2 (p0 + 1), ..., 2 p1 (every later range starts inside
// the request, so its segment of b is that range's first).
struct ReqSplit {
  int32_t p0, p1, first_odd, pad;
};

struct PlanHeader {
  int32_t total_units;  // U
  int32_t num_ranges;   // P (0 when U == 0)
  int32_t max_ranges;   // P_max the plan was made for
  int32_t batch;
  int32_t unit_tokens;
  int32_t max_blocks_per_seq;
  int32_t block_size;
  int32_t pad;
};

// Workspace layout (all offsets 256-byte aligned):
//   PlanHeader
//   int32 seq_len[B]          clamped lengths
//   int32 unit_prefix[B + 1]  U_b
//   int32 range_start[P_max + 1]  R_p (entries past P hold U)
//   int32 range_first[P_max]  first request with units in range p
//   int64 cost_prefix[B + 1]  cost before request b (planner scratch)
//   int32 counters[B * 2]     split arrival counters (left at zero)
//   int32 seg_count[P_max]    segments of range p (0 for p >= P)
//   SegRec seg_rec[P_max][kSegCache]
//   ReqSplit req_split[B]
//   fp32 lse_part[2 * P_max * H]
//   bf16 o_part[2 * P_max][512 / 8][H][8]   (a partial: the segment's output
//                                            normalised by its own sum, in the
//                                            output's type; one partial's heads
//                                            of eight dims are contiguous)
struct WorkspaceLayout {
  size_t seq_len, unit_prefix, range_start, range_first, cost_prefix, counters, seg_count, seg_rec, req_split, lse_part,
      o_part, total;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

__host__ __device__ inline WorkspaceLayout workspace_layout(int batch, int heads, int max_ranges) {
  WorkspaceLayout w;
  size_t o = align256(sizeof(PlanHeader));
  w.seq_len = o;      o = align256(o + sizeof(int32_t) * (size_t)batch);
  w.unit_prefix = o;  o = align256(o + sizeof(int32_t) * ((size_t)batch + 1));
  w.range_start = o;  o = align256(o + sizeof(int32_t) * ((size_t)max_ranges + 1));
  w.range_first = o;  o = align256(o + sizeof(int32_t) * ((size_t)max_ranges + 1));
  w.cost_prefix = o;  o = align256(o + sizeof(int64_t) * ((size_t)batch + 1));
  w.counters = o;     o = align256(o + sizeof(int32_t) * 2 * (size_t)batch);
  w.seg_count = o;    o = align256(o + sizeof(int32_t) * (size_t)max_ranges);
  w.seg_rec = o;      o = align256(o + sizeof(SegRec) * kSegCache * (size_t)max_ranges);
  w.req_split = o;    o = align256(o + sizeof(ReqSplit) * (size_t)batch);
  w.lse_part = o;     o = align256(o + sizeof(float) * 2 * (size_t)max_ranges * heads);
  w.o_part = o;       o = align256(o + sizeof(__nv_bfloat16) * 2 * (size_t)max_ranges * heads * kVDim);
  w.total = o;
  return w;
}

struct PlanView {
  const PlanHeader *hdr;
  const int32_t *seq_len;
  const int32_t *unit_prefix;
  const int32_t *range_start;
  const int32_t *range_first;
  const int64_t *cost_prefix;
  int32_t *counters;
  const int32_t *seg_count;
  const SegRec *seg_rec;
  const ReqSplit *req_split;
  float *lse_part;
  __nv_bfloat16 *o_part;
};

__host__ __device__ inline PlanView plan_view(void *ws, int batch, int heads, int max_ranges) {
  WorkspaceLayout l = workspace_layout(batch, heads, max_ranges);
  char *b = (char *)ws;
  PlanView v;
  v.hdr = (const PlanHeader *)b;
  v.seq_len = (const int32_t *)(b + l.seq_len);
  v.unit_prefix = (const int32_t *)(b + l.unit_prefix);
  v.range_start = (const int32_t *)(b + l.range_start);
  v.range_first = (const int32_t *)(b + l.range_first);
  v.cost_prefix = (const int64_t *)(b + l.cost_prefix);
  v.counters = (int32_t *)(b + l.counters);
  v.seg_count = (const int32_t *)(b + l.seg_count);
  v.seg_rec = (const SegRec *)(b + l.seg_rec);
  v.req_split = (const ReqSplit *)(b + l.req_split);
  v.lse_part = (float *)(b + l.lse_part);
  v.o_part = (__nv_bfloat16 *)(b + l.o_part);
  return v;
}

// Segments of range p, in plan order: request b, tokens [t0, t1), partial
// slot (-1: the request is not split).  The first kSegCache come from the
// plan's records (one memory round trip); later ones, for ranges that cross
// many short requests, by walking the plan on from the last request.
// kUnitTokens is the plan's unit (the decode kernels' tile).
template <int kUnitTokens>
struct SegIter {
  PlanView v;
  int32_t batch, p, n, idx, b;
  int32_t row0;  // cache row of the current segment's first token, -1 if unknown
  SegRec first;  // record 0, loaded together with the count
  // n_ and first_: the range's segment count and first record, loaded by the
  // caller at kernel entry (one round trip for both, overlapping the setup)
  __device__ void init(const PlanView &pv, int32_t batch_, int32_t p_, int32_t n_,
                       const SegRec &first_) {
    v = pv;
    batch = batch_;
    p = p_;
    n = n_;
    first = first_;
    idx = 0;
    b = -1;
    row0 = -1;
  }
  __device__ bool next(int32_t &t0, int32_t &t1, int32_t &slot) {
    if (idx >= n) return false;
    if (idx < kSegCache) {
      const SegRec r = idx == 0 ? first : v.seg_rec[(int64_t)p * kSegCache + idx];
      ++idx;
      b = r.b;
      t0 = r.t0;
      t1 = r.t1;
      slot = r.slot;
      row0 = r.row0;
      return true;
    }
    row0 = -1;
    const int32_t r0 = v.range_start[p], r1 = v.range_start[p + 1];
    // from the request after the last record's (which a plan made for other
    // arguments may have left anywhere: the walk stays within [0, batch))
    for (b = (b >= -1 && b < batch) ? b + 1 : batch; b < batch; ++b) {
      const int32_t Ub = v.unit_prefix[b];
      if (Ub >= r1) return false;
      const int32_t Ue = v.unit_prefix[b + 1];
      const int32_t u0 = max(r0, Ub), u1 = min(r1, Ue);
      if (u0 >= u1) continue;
      t0 = (u0 - Ub) * kUnitTokens;
      t1 = min((u1 - Ub) * kUnitTokens, v.seq_len[b]);
      slot = segment_slot(p, r0, r1, Ub, Ue);
      ++idx;
      return true;
    }
    return false;
  }
};

// Whether a range's first record (loaded by every thread at kernel entry)
// belongs to a plan made for these arguments: it carries their stamp and
// keeps within the request, the block table and the partial slots.  A plan
// that passes is the one these arguments make, so its other records and
// arrays are valid too.  Checked once per CTA, before any role reads the
// plan further (a check inside the segment walk, inlined in every role,
// measured slower).  A range with no segments reads nothing.
__device__ __forceinline__ bool plan_record_ok(int32_t seg_n, const SegRec &r, int32_t stamp,
                                               int32_t batch, int32_t max_len,
                                               int32_t num_slots) {
  return seg_n <= 0 || (r.stamp == stamp && r.b >= 0 && r.b < batch && r.t0 >= 0 &&
                        r.t0 < r.t1 && r.t1 <= max_len && r.slot >= -1 && r.slot < num_slots);
}


}  // namespace mla
