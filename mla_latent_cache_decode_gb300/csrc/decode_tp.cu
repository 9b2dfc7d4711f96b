// Tensor-core MLA decode for few heads (sm_103a): a tensor-parallel rank's
// share of the 128 heads.
//
// What is computed: the absorbed-form MLA decode of decode_tc.cu for H <= 32
// heads.  Every head's score uses all 576 dims of each cached row (512 kv_c +
// 64 k_rope shared by all heads) and its output is the softmax-weighted sum of
// the 512-dim kv_c.  Under tensor-parallel attention a rank owns 128 / TP of
// the heads (16 at TP = 8) yet reads every cached row of every request, since
// all heads share the latent [dp-attention-expert-parallel-mla-kv-replication
// (inferenceinterviews.com), "A strong answer": 45.8 GB per GPU per step at
// TP = 8; MLA 的 TP 切分 (10100.com), section 3.1].
//
// Transposed products.  With so few heads S = Q K^T has M = H rows, below the
// tensor core's smallest M, so the kernel puts tokens and value dims in M and
// the heads in N:
//   S^T [64 tokens x H]  = K [64 x 576] . Q^T              (M = 64, 36 MMAs)
//   O^T [512 dims x H]  += V^T [512 x 64] . P^T [64 x H]   (4 blocks of M = 128)
// V is the first 512 dims of the tile's rows, read in place: K-major as the A
// operand of S^T, MN-major as the A operand of O^T.  Q and P^T are the B
// operands (K-major).  H is padded to kHP = 16 or 32 (N of an M = 128 MMA is a
// multiple of 16); pad heads read other rows of q (zeros past its end) and
// are never stored, and no head's result depends on another head's.
//
// Layout of the work.  One CTA per SM and one split range of the plan (64-token
// units, common.cuh) per CTA.  A tile is 64 tokens of all 576 dims, 72 KB in
// nine 64-dim chunks with the 128-byte swizzle, fetched (when a page holds 64
// tokens or more) by three 3-D TMA boxes: value dims 0-255 and 256-511 into a
// ring of 32 KB halves, each freed once its two O^T blocks are done, and the
// rope chunk into a ring of its own, freed once the scores are.  Tensor memory
// holds O^T (four blocks of kHP columns, all 128 lanes: lane = value dim) and
// two S^T buffers of kHP columns (an M = 64 result puts rows 16q .. 16q + 15
// in lanes 32q .. 32q + 15).
//
// Softmax.  A tile's tokens lie across threads (lanes 0-15 of the four
// softmax warps), so a head's tile max is a reduction across threads: each
// warp reduces its 16 tokens per head by a shuffle transpose, the four warps'
// results meet in shared memory, and every thread then holds the same
// running max of every head (lazy rescale of O^T, as in decode_tc.cu).  Sums
// stay per thread until the segment ends.
//
// Warp roles: 0 loads tiles; 1 issues the S^T MMAs; 2 issues the O^T MMAs;
// 3 loads each segment's Q and owns the tensor memory; 4-7 run the softmax
// (thread = token) and the epilogue (thread = value dim of each O^T block).
// Every wait is bounded; one that runs out reports MLA_ERR_DEVICE_TIMEOUT and
// raises the CTA's abort flag, which ends the other roles' waits.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "sm100.cuh"
#include "tmap.h"

namespace mla {
namespace tp {

using namespace sm100;

constexpr int kTile = 64;                   // tokens per tile (= plan unit)
constexpr int kChunks = kRow / 64;          // 9 chunks of 64 dims per row
constexpr int kChunkBytes = kTile * 128;    // 8 KB: 64 tokens x 64 dims
constexpr int kHalfChunks = 4;              // a value half: 256 dims
constexpr int kHalfBytes = kHalfChunks * kChunkBytes;  // 32 KB
constexpr int kRopeSlots = 2;
constexpr int kQBufs = 2;                   // the next segment's Q loads early
constexpr int kThreads = 256;
constexpr int kSoftmaxWarp0 = 4;
constexpr uint64_t kWaitBudgetNs = 100000000ull;  // 100 ms per wait, far above any legal wait
constexpr uint64_t kDrainBudgetNs = 10000000ull;  // 10 ms to drain in-flight copies on abort
constexpr float kRescaleThreshold = 8.0f;         // log2 units

// Ring slots of value halves: as many as shared memory holds beside the rope
// ring, two Q buffers and P^T (5 at 16 heads: 2.5 tiles of values in flight).
template <int kHP>
constexpr int half_slots() {
  return kHP == 16 ? 5 : 4;
}

// A tile arrives as three boxes with their own barriers: value dims 0-255
// (half 0, chunks 0-3), 256-511 (half 1, chunks 4-7) and the rope (chunk 8).
// The halves share one ring and the rope has its own, because they are freed
// at different times: a half once the O^T MMAs of its two blocks are done,
// the rope once the tile's S^T MMAs are.  Half h of tile g is the ring's
// item 2g + h.
template <int kHP>
struct __align__(1024) Smem {
  uint8_t kv[half_slots<kHP>()][kHalfBytes];  // chunk c of a half at + 8 KB c, token r at + 128 r
  uint8_t rope[kRopeSlots][kChunkBytes];
  uint8_t q[kQBufs][kChunks][kHP * 128];      // Q of a segment: chunk c = kHP heads x 64 dims
  uint8_t p[2][kHP * 128];                    // P^T of a tile: row h = the tile's 64 tokens (bf16)
  float red[2][kHP][4];                       // each softmax warp's tile max of every head
  float redl[kHP][4];                         // each softmax warp's sum of every head
  uint64_t kv_full[half_slots<kHP>()], kv_empty[half_slots<kHP>()];
  uint64_t rope_full[kRopeSlots], rope_empty[kRopeSlots];
  uint64_t q_full[kQBufs], q_free[kQBufs];
  // S^T buffer written / read by all softmax warps; P^T written; O^T MMAs of
  // the tile done; the four warps' maxima (sums) in red (redl)
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2], red_full[2], redl_full;
  uint64_t fin_s, fin_pv, roles_done;
  uint32_t tmem_base;
  int abort;
};

// 227 KB of dynamic shared memory per CTA, with 1 KB for the alignment
static_assert(sizeof(Smem<16>) + 1024 <= 232448 && sizeof(Smem<32>) + 1024 <= 232448,
              "shared memory");

template <int kHP>
constexpr uint32_t tmem_cols() {
  return 6 * kHP <= 128 ? 128u : 256u;  // O^T (4 kHP) + two S^T buffers (2 kHP)
}

struct Maps {
  CUtensorMap kv4;   // {64, rows, 9 chunks}, box {64, 64, 4}: value dims of a tile part
  CUtensorMap kv1;   // the same view, box {64, 64, 1}: the rope chunk
  CUtensorMap kv2d;  // {576, rows}, box {64, block_size}: one chunk of one page
  CUtensorMap q;     // {64, batch * heads, 9 chunks}, box {64, kHP, 9}
};

struct Params {
  const int32_t *block_table;
  int32_t max_blocks_per_seq;
  int32_t block_size;
  int32_t num_blocks;
  int32_t batch;
  int32_t heads;
  float scale_log2;
  __nv_bfloat16 *out;
  float *lse;
  void *ws;
  int32_t max_ranges;
  int32_t *dev_status;
};

template <int kHP>
__device__ __forceinline__ void set_abort(Smem<kHP> &s, int32_t *dev_status) {
  s.abort = 1;
  report(dev_status, MLA_ERR_DEVICE_TIMEOUT);
}

// Every lane polls, then the warp agrees (uniform control flow around the
// warp-collective tcgen05 instructions).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const volatile int *abort) {
  const bool ok = mbar_wait(bar, parity, abort, kWaitBudgetNs);
  return __all_sync(0xffffffffu, ok);
}

// Reduces v[i] across lanes 0-15 (and, separately, across lanes 16-31) for
// every i < kN: a shuffle transpose that halves the values each step, so lane
// l ends with the results for i in [l kN/16, (l + 1) kN/16) (l < 16) in
// v[0 .. kN/16).
template <int kN, bool kMax>
__device__ __forceinline__ void transpose_reduce16(float (&v)[kN], int lane) {
#pragma unroll
  for (int step = 0; step < 4; ++step) {
    const int o = 8 >> step;
    const int half = kN >> (step + 1);
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int k = 0; k < half; ++k) {
      const float send = upper ? v[k] : v[k + half];
      const float keep = upper ? v[k + half] : v[k];
      const float recv = __shfl_xor_sync(0xffffffffu, send, o);
      v[k] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
}

template <int kHP>
__device__ __forceinline__ void tmem_ld_heads(uint32_t taddr, uint32_t (&r)[kHP]) {
  if constexpr (kHP == 16) tmem_ld16(taddr, r); else tmem_ld32(taddr, r);
}
template <int kHP>
__device__ __forceinline__ void tmem_st_heads(uint32_t taddr, const uint32_t (&r)[kHP]) {
  if constexpr (kHP == 16) tmem_st16(taddr, r); else tmem_st32(taddr, r);
}

template <int kHP>
__global__ void __launch_bounds__(kThreads, 1)
    decode_tp_kernel(const __grid_constant__ Maps maps, const Params prm) {
  constexpr uint32_t kColO = 0, kColS = 4 * kHP, kCols = tmem_cols<kHP>();
  constexpr int kQBytes = kChunks * kHP * 128;
  constexpr int kHalves = half_slots<kHP>();
  extern __shared__ uint8_t smem_raw[];
  Smem<kHP> &s = *reinterpret_cast<Smem<kHP> *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int range = blockIdx.x;  // this CTA's split range
  const PlanView v = plan_view(prm.ws, prm.batch, prm.heads, prm.max_ranges);
  const volatile int *abort_flag = &s.abort;
  const int32_t seg_n = v.seg_count[range];
  const SegRec seg_first = v.seg_rec[(int64_t)range * kSegCache];

  if (tid == 0) {
    for (int i = 0; i < kHalves; ++i) {
      mbar_init(smem_u32(&s.kv_full[i]), 1);
      mbar_init(smem_u32(&s.kv_empty[i]), 1);
    }
    for (int i = 0; i < kRopeSlots; ++i) {
      mbar_init(smem_u32(&s.rope_full[i]), 1);
      mbar_init(smem_u32(&s.rope_empty[i]), 1);
    }
    for (int i = 0; i < kQBufs; ++i) {
      mbar_init(smem_u32(&s.q_full[i]), 1);
      mbar_init(smem_u32(&s.q_free[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s.s_full[i]), 1);
      mbar_init(smem_u32(&s.s_free[i]), 4);
      mbar_init(smem_u32(&s.p_full[i]), 4);
      mbar_init(smem_u32(&s.pv_done[i]), 1);
      mbar_init(smem_u32(&s.red_full[i]), 4);
    }
    mbar_init(smem_u32(&s.redl_full), 4);
    mbar_init(smem_u32(&s.fin_s), 1);
    mbar_init(smem_u32(&s.fin_pv), 1);
    mbar_init(smem_u32(&s.roles_done), kThreads / 32);
    s.abort = 0;
    fence_mbarrier_init_cluster();
  }
  if (warp == 3) {
    tmem_alloc(smem_u32(&s.tmem_base), kCols);
    tmem_relinquish();
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  const bool active = seg_n > 0;
  // Whether the plan was made for these arguments (see plan_record_ok),
  // checked by the roles that form global addresses from its records, at
  // their first record: the tile producer (block-table reads; it reports a
  // plan made for other arguments and raises the abort flag, which ends the
  // other roles) and the softmax (output writes).
  const int32_t seg_stamp =
      plan_stamp(prm.batch, prm.max_ranges, kTile, prm.block_size, prm.max_blocks_per_seq);
  auto plan_ok = [&]() {
    return plan_record_ok(seg_n, seg_first, seg_stamp, prm.batch,
                          prm.max_blocks_per_seq * prm.block_size, 2 * prm.max_ranges);
  };
  const int BS = prm.block_size;
  const bool big_pages = BS >= kTile;  // a tile lies inside one page: one box

  if (warp == 0) {
    // ------------------------------------------------------------ tile loads
    if (active && elect_one_sync()) {
      const bool plan_good = plan_ok();
      if (!plan_good) {
        s.abort = 1;
        report(prm.dev_status, MLA_ERR_DEVICE_PLAN);
      }
      SegIter<kTile> it;
      it.init(v, prm.batch, range, seg_n, seg_first);
      int32_t t0, t1, slot_p;
      uint32_t g = 0;
      uint32_t half_issued[kHalves] = {}, rope_issued[kRopeSlots] = {};
      const int box_rows = big_pages ? kTile : BS;
      const int64_t nb = prm.num_blocks;
      if (big_pages) {
        prefetch_tmap(&maps.kv4);
        prefetch_tmap(&maps.kv1);
      } else {
        prefetch_tmap(&maps.kv2d);
      }
      bool ok = plan_good;
      while (ok && it.next(t0, t1, slot_p)) {
        const int32_t *row = prm.block_table + (int64_t)it.b * prm.max_blocks_per_seq;
        for (int32_t tt = t0; tt < t1; tt += kTile, ++g) {
          const int nbx = big_pages ? 1 : (min(kTile, t1 - tt) + BS - 1) / BS;
          // cache rows of the tile's boxes, looked up before the slot wait so
          // that the table loads overlap it
          int32_t y[kTile / 16];
          if (tt == t0 && it.row0 >= 0 && big_pages) {
            y[0] = it.row0;
          } else {
#pragma unroll
            for (int j = 0; j < kTile / 16; ++j) {
              if (j >= nbx) break;
              int32_t blk = row[(tt + j * box_rows) / BS];
              if (blk < 0 || blk >= nb) {
                report(prm.dev_status, MLA_ERR_DEVICE_RANGE);
                blk = 0;
              }
              y[j] = blk * BS + (tt + j * box_rows) % BS;
            }
          }
          // the two value halves, then the rope, each once its slot is free
          for (int hf = 0; hf < 2; ++hf) {
            const uint32_t k = 2 * g + hf;
            const int sl = k % kHalves;
            if (!mbar_wait(smem_u32(&s.kv_empty[sl]), ((k / kHalves) & 1u) ^ 1u, abort_flag,
                           kWaitBudgetNs)) {
              set_abort(s, prm.dev_status);
              ok = false;
              break;
            }
            const uint32_t bar = smem_u32(&s.kv_full[sl]);
            mbar_arrive_expect_tx(bar, (uint32_t)(kHalfChunks * nbx * box_rows * 128));
            if (big_pages) {
              tma_load_3d(smem_u32(s.kv[sl]), &maps.kv4, 0, y[0], kHalfChunks * hf, bar);
            } else {
#pragma unroll
              for (int j = 0; j < kTile / 16; ++j) {
                if (j >= nbx) break;
                for (int c = 0; c < kHalfChunks; ++c)
                  tma_load_2d(smem_u32(s.kv[sl]) + c * kChunkBytes + j * box_rows * 128,
                              &maps.kv2d, 64 * (kHalfChunks * hf + c), y[j], bar);
              }
            }
            ++half_issued[sl];
          }
          if (!ok) break;
          const int rs = g % kRopeSlots;
          if (!mbar_wait(smem_u32(&s.rope_empty[rs]), ((g / kRopeSlots) & 1u) ^ 1u, abort_flag,
                         kWaitBudgetNs)) {
            set_abort(s, prm.dev_status);
            ok = false;
            break;
          }
          const uint32_t rbar = smem_u32(&s.rope_full[rs]);
          mbar_arrive_expect_tx(rbar, (uint32_t)(nbx * box_rows * 128));
          if (big_pages) {
            tma_load_3d(smem_u32(s.rope[rs]), &maps.kv1, 0, y[0], kChunks - 1, rbar);
          } else {
#pragma unroll
            for (int j = 0; j < kTile / 16; ++j) {
              if (j >= nbx) break;
              tma_load_2d(smem_u32(s.rope[rs]) + j * box_rows * 128, &maps.kv2d,
                          64 * (kChunks - 1), y[j], rbar);
            }
          }
          ++rope_issued[rs];
        }
      }
      if (s.abort) {  // let the loads in flight land before exit
        for (int i = 0; i < kHalves; ++i)
          if (half_issued[i] > 0)
            (void)mbar_wait(smem_u32(&s.kv_full[i]), (half_issued[i] - 1) & 1u, nullptr,
                            kDrainBudgetNs);
        for (int i = 0; i < kRopeSlots; ++i)
          if (rope_issued[i] > 0)
            (void)mbar_wait(smem_u32(&s.rope_full[i]), (rope_issued[i] - 1) & 1u, nullptr,
                            kDrainBudgetNs);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ S^T = K Q^T
    if (active && elect_one_sync()) {
      SegIter<kTile> it;
      it.init(v, prm.batch, range, seg_n, seg_first);
      int32_t t0, t1, slot_p;
      uint32_t g = 0, seg = 0;
      const uint32_t id = idesc_bf16_f32(64, kHP, 0);
      // descriptors of slot 0 chunk 0 / Q buffer 0 chunk 0; slots, chunks and
      // k-steps add their byte offset >> 4 to the start-address field (no
      // carry: every shared-memory address here is below 2^18)
      const uint64_t d_kv = smem_desc(smem_u32(s.kv[0]), 16, 1024, kSwizzle128B);
      const uint64_t d_rope = smem_desc(smem_u32(s.rope[0]), 16, 1024, kSwizzle128B);
      const uint64_t d_q = smem_desc(smem_u32(s.q[0][0]), 16, 1024, kSwizzle128B);
      bool ok = true;
      while (ok && it.next(t0, t1, slot_p)) {
        const int qb = seg % kQBufs;
        if (!mbar_wait(smem_u32(&s.q_full[qb]), (seg / kQBufs) & 1u, abort_flag, kWaitBudgetNs)) {
          set_abort(s, prm.dev_status);
          break;
        }
        ++seg;
        for (int32_t tt = t0; tt < t1; tt += kTile, ++g) {
          // the S^T buffer was last read by the softmax of tile g - 2
          if (g >= 2 && !mbar_wait(smem_u32(&s.s_free[g & 1u]), ((g >> 1) - 1) & 1u, abort_flag,
                                   kWaitBudgetNs)) {
            set_abort(s, prm.dev_status);
            ok = false;
            break;
          }
          const uint32_t d_s = tmem + kColS + kHP * (g & 1u);
          const uint64_t b0 = d_q + (uint64_t)((qb * kQBytes) >> 4);
          for (int hf = 0; hf < 2 && ok; ++hf) {
            const uint32_t k = 2 * g + hf;
            const int sl = k % kHalves;
            if (!mbar_wait(smem_u32(&s.kv_full[sl]), (k / kHalves) & 1u, abort_flag,
                           kWaitBudgetNs)) {
              set_abort(s, prm.dev_status);
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t a0 = d_kv + (uint64_t)((sl * kHalfBytes) >> 4);
#pragma unroll
            for (int c = 0; c < kHalfChunks; ++c) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_ss(d_s, a0 + (uint64_t)((c * kChunkBytes + kk * 32) >> 4),
                       b0 + (uint64_t)((((kHalfChunks * hf + c) * kHP * 128) + kk * 32) >> 4), id,
                       (hf | c | kk) ? 1u : 0u);
            }
          }
          if (!ok) break;
          const int rs = g % kRopeSlots;
          if (!mbar_wait(smem_u32(&s.rope_full[rs]), (g / kRopeSlots) & 1u, abort_flag,
                         kWaitBudgetNs)) {
            set_abort(s, prm.dev_status);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t r0 = d_rope + (uint64_t)((rs * kChunkBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(d_s, r0 + (uint64_t)((kk * 32) >> 4),
                   b0 + (uint64_t)((((kChunks - 1) * kHP * 128) + kk * 32) >> 4), id, 1u);
          mma_commit(smem_u32(&s.s_full[g & 1u]));
          mma_commit(smem_u32(&s.rope_empty[rs]));  // the rope is read by S^T only
        }
        if (!ok) break;
        mma_commit(smem_u32(&s.q_free[qb]));  // this segment's Q is no longer read
      }
      mma_commit(smem_u32(&s.fin_s));
      if (!mbar_wait(smem_u32(&s.fin_s), 0, nullptr, kWaitBudgetNs))
        report(prm.dev_status, MLA_ERR_DEVICE_TIMEOUT);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ O^T += V^T P^T
    if (active && elect_one_sync()) {
      SegIter<kTile> it;
      it.init(v, prm.batch, range, seg_n, seg_first);
      int32_t t0, t1, slot_p;
      uint32_t g = 0;
      const uint32_t id = idesc_bf16_f32(128, kHP, 0, 1);  // A (V^T) MN-major
      // V^T: M = 128 dims of two adjacent chunks (LBO: chunk stride), K = tokens
      const uint64_t d_v = smem_desc(smem_u32(s.kv[0]), kChunkBytes, 1024, kSwizzle128B);
      const uint64_t d_p = smem_desc(smem_u32(s.p[0]), 16, 1024, kSwizzle128B);
      bool ok = true;
      while (ok && it.next(t0, t1, slot_p)) {
        for (int32_t tt = t0; tt < t1; tt += kTile, ++g) {
          if (!mbar_wait(smem_u32(&s.p_full[g & 1u]), (g >> 1) & 1u, abort_flag, kWaitBudgetNs)) {
            set_abort(s, prm.dev_status);
            ok = false;
            break;
          }
          tc_fence_after();
          const int ksteps = (min(kTile, t1 - tt) + 15) >> 4;
          const uint64_t b0 = d_p + (uint64_t)(((g & 1u) * kHP * 128) >> 4);
          // block i = 2 hf + ib: value dims 128 i .. 128 i + 127, chunks 2 ib and
          // 2 ib + 1 of half hf; the half's slot is free once its blocks are done
          for (int hf = 0; hf < 2; ++hf) {
            const int sl = (2 * g + hf) % kHalves;
            const uint64_t a0 = d_v + (uint64_t)((sl * kHalfBytes) >> 4);
#pragma unroll
            for (int ib = 0; ib < 2; ++ib) {
              for (int kt = 0; kt < ksteps; ++kt)
                mma_ss(tmem + kColO + (2 * hf + ib) * kHP,
                       a0 + (uint64_t)((2 * ib * kChunkBytes + kt * 2048) >> 4),
                       b0 + (uint64_t)((kt * 32) >> 4), id, (tt > t0 || kt > 0) ? 1u : 0u);
            }
            mma_commit(smem_u32(&s.kv_empty[sl]));
          }
          mma_commit(smem_u32(&s.pv_done[g & 1u]));
        }
      }
      mma_commit(smem_u32(&s.fin_pv));
      if (!mbar_wait(smem_u32(&s.fin_pv), 0, nullptr, kWaitBudgetNs))
        report(prm.dev_status, MLA_ERR_DEVICE_TIMEOUT);
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ Q loads
    // Each segment's Q into the next buffer, once the S^T MMAs of the segment
    // that used it before are done.
    if (active && elect_one_sync()) {
      SegIter<kTile> it;
      it.init(v, prm.batch, range, seg_n, seg_first);
      int32_t t0, t1, slot_p;
      uint32_t seg = 0;
      uint32_t issued[kQBufs] = {0, 0};
      prefetch_tmap(&maps.q);
      while (it.next(t0, t1, slot_p)) {
        const int qb = seg % kQBufs;
        if (!mbar_wait(smem_u32(&s.q_free[qb]), ((seg / kQBufs) & 1u) ^ 1u, abort_flag,
                       kWaitBudgetNs)) {
          set_abort(s, prm.dev_status);
          break;
        }
        mbar_arrive_expect_tx(smem_u32(&s.q_full[qb]), (uint32_t)kQBytes);
        tma_load_3d(smem_u32(s.q[qb][0]), &maps.q, 0, it.b * prm.heads, 0,
                    smem_u32(&s.q_full[qb]));
        ++issued[qb];
        ++seg;
      }
      if (s.abort) {
        for (int i = 0; i < kQBufs; ++i)
          if (issued[i] > 0)
            (void)mbar_wait(smem_u32(&s.q_full[i]), (issued[i] - 1) & 1u, nullptr, kDrainBudgetNs);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    const int q4 = warp - kSoftmaxWarp0;  // TMEM lane quadrant (= warp % 4)
    const int st = tid - kSoftmaxWarp0 * 32;
    const bool tok_lane = lane < 16;      // an M = 64 row lives in lanes 0-15 of a quadrant
    const int t = 16 * q4 + lane;         // this lane's token in a tile (tok_lane)
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    const int H = prm.heads;
    const float c = prm.scale_log2;

    // requests with no context: out = 0, lse = -inf
    for (int b = range; b < prm.batch; b += (int)gridDim.x) {
      if (v.seq_len[b] != 0) continue;
      uint4 *o = reinterpret_cast<uint4 *>(prm.out + (int64_t)b * H * kVDim);
      for (int k = st; k < H * (kVDim / 8); k += 128) o[k] = make_uint4(0, 0, 0, 0);
      if (prm.lse && st < H) prm.lse[(int64_t)b * H + st] = -INFINITY;
    }

    if (active && plan_ok()) {  // outputs are written where the plan's records say
      SegIter<kTile> it;
      it.init(v, prm.batch, range, seg_n, seg_first);
      int32_t t0, t1, slot_p;
      uint32_t g = 0, seg = 0;
      bool ok = true;
      float m_used[kHP], l_part[kHP];
      while (ok && it.next(t0, t1, slot_p)) {
        const int b = it.b;
        for (int32_t tt = t0; tt < t1; tt += kTile, ++g) {
          const int n = min(kTile, t1 - tt);
          const bool first = (tt == t0);
          if (!warp_wait(smem_u32(&s.s_full[g & 1u]), (g >> 1) & 1u, abort_flag)) {
            if (lane == 0) set_abort(s, prm.dev_status);
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t xr[kHP];
          tmem_ld_heads<kHP>(lane_base + kColS + kHP * (g & 1u), xr);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&s.s_free[g & 1u]));
          const bool valid = tok_lane && t < n;
          float x[kHP], mx[kHP];
#pragma unroll
          for (int h = 0; h < kHP; ++h) {
            x[h] = valid ? __uint_as_float(xr[h]) : -INFINITY;
            mx[h] = x[h];
          }
          // the tile max of every head: 16 tokens per warp, then the four warps
          transpose_reduce16<kHP, true>(mx, lane);
          if (tok_lane) {
#pragma unroll
            for (int j = 0; j < kHP / 16; ++j) s.red[g & 1u][lane * (kHP / 16) + j][q4] = mx[j];
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&s.red_full[g & 1u]));
          if (!warp_wait(smem_u32(&s.red_full[g & 1u]), (g >> 1) & 1u, abort_flag)) {
            if (lane == 0) set_abort(s, prm.dev_status);
            ok = false;
            break;
          }
          // every thread takes the same decisions from the same maxima
          float alpha[kHP];
          bool rescale = false;
#pragma unroll
          for (int h = 0; h < kHP; ++h) {
            const float4 r = *reinterpret_cast<const float4 *>(&s.red[g & 1u][h][0]);
            const float tm = fmaxf(fmaxf(r.x, r.y), fmaxf(r.z, r.w)) * c;
            alpha[h] = 1.f;
            if (first) {
              m_used[h] = tm;
              l_part[h] = 0.f;
            } else if (tm > m_used[h] + kRescaleThreshold) {
              alpha[h] = ex2_approx(m_used[h] - tm);
              m_used[h] = tm;
              rescale = true;
            }
          }
          float pr[kHP];
#pragma unroll
          for (int h = 0; h < kHP; ++h) {
            pr[h] = valid ? ex2_approx(fmaf(x[h], c, -m_used[h])) : 0.f;
            l_part[h] = l_part[h] * alpha[h] + pr[h];
          }
          if (rescale) {
            // O^T may be rescaled only once the previous tile's O^T MMAs are done
            if (!warp_wait(smem_u32(&s.pv_done[(g - 1) & 1u]), ((g - 1) >> 1) & 1u, abort_flag)) {
              if (lane == 0) set_abort(s, prm.dev_status);
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int i = 0; i < 4; ++i) {
              uint32_t o[kHP];
              tmem_ld_heads<kHP>(lane_base + kColO + i * kHP, o);
              tmem_wait_ld();
#pragma unroll
              for (int h = 0; h < kHP; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[h]);
              tmem_st_heads<kHP>(lane_base + kColO + i * kHP, o);
            }
            tmem_wait_st();
          }
          // the P^T buffer was last read by the O^T MMAs of tile g - 2
          if (g >= 2 &&
              !warp_wait(smem_u32(&s.pv_done[g & 1u]), ((g >> 1) - 1) & 1u, abort_flag)) {
            if (lane == 0) set_abort(s, prm.dev_status);
            ok = false;
            break;
          }
          // The O^T MMAs of a tail tile read tokens [0, ceil16(n)); rows past the
          // sequence end hold whatever the page held (maybe NaN; 0 * NaN = NaN),
          // so zero them in the eight value chunks (whole 128-byte rows).
          if (n & 15) {
            const int rows = ((n + 15) & ~15) - n;
            for (int k = st; k < rows * 64; k += 128) {
              const int r = n + (k >> 6), ch = (k >> 3) & 7, u = k & 7;
              uint8_t *half = s.kv[(2 * g + (ch >> 2)) % kHalves];
              *reinterpret_cast<uint4 *>(half + (ch & 3) * kChunkBytes + r * 128 + u * 16) =
                  make_uint4(0, 0, 0, 0);
            }
          }
          // P^T in bf16, K-major with the 128-byte swizzle: row h = head h,
          // token t at 16-byte unit (t / 8) ^ (h % 8)
          if (tok_lane) {
            uint8_t *pb = s.p[g & 1u];
#pragma unroll
            for (int h = 0; h < kHP; ++h)
              *reinterpret_cast<__nv_bfloat16 *>(pb + h * 128 + ((((t >> 3) ^ (h & 7))) << 4) +
                                                 (t & 7) * 2) = __float2bfloat16_rn(pr[h]);
          }
          fence_proxy_async_shared();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&s.p_full[g & 1u]));
        }
        if (!ok) break;
        // ---- epilogue: the segment's sums, then O^T / l after its last MMAs
        transpose_reduce16<kHP, false>(l_part, lane);
        if (tok_lane) {
#pragma unroll
          for (int j = 0; j < kHP / 16; ++j) s.redl[lane * (kHP / 16) + j][q4] = l_part[j];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s.redl_full));
        const uint32_t gl = g - 1;
        if (!warp_wait(smem_u32(&s.redl_full), seg & 1u, abort_flag) ||
            !warp_wait(smem_u32(&s.pv_done[gl & 1u]), (gl >> 1) & 1u, abort_flag)) {
          if (lane == 0) set_abort(s, prm.dev_status);
          break;
        }
        ++seg;
        tc_fence_after();
        float inv[kHP];
        float lse_val = -INFINITY;
#pragma unroll
        for (int h = 0; h < kHP; ++h) {
          const float4 r = *reinterpret_cast<const float4 *>(&s.redl[h][0]);
          const float l = (r.x + r.y) + (r.z + r.w);
          inv[h] = 1.f / l;
          if (h == st) lse_val = (m_used[h] + log2f(l)) * 0.69314718055994531f;
        }
        // thread = value dim 128 i + 32 q4 + lane of block i; a warp's 32 dims
        // of one head are 64 contiguous bytes
        __nv_bfloat16 *dst = slot_p < 0 ? prm.out + (int64_t)b * H * kVDim
                                        : v.o_part + (int64_t)slot_p * H * kVDim;
#pragma unroll 1
        for (int i = 0; i < 4; ++i) {
          uint32_t o[kHP];
          tmem_ld_heads<kHP>(lane_base + kColO + i * kHP, o);
          tmem_wait_ld();
          const int d = 128 * i + 32 * q4 + lane;
#pragma unroll
          for (int h = 0; h < kHP; ++h)
            if (h < H) dst[(int64_t)h * kVDim + d] = __float2bfloat16_rn(__uint_as_float(o[h]) * inv[h]);
        }
        if (st < H) {
          if (slot_p < 0) {
            if (prm.lse) prm.lse[(int64_t)b * H + st] = lse_val;
          } else {
            v.lse_part[(int64_t)slot_p * H + st] = lse_val;
          }
        }
        tc_fence_before();
      }
    }
  }

  // ------------------------------------------------------------ teardown
  // Each warp reports the end of its role once all its lanes are here, and
  // the tensor memory is freed only after every report.
  __syncwarp();
  tc_fence_before();
  if (lane == 0) mbar_arrive(smem_u32(&s.roles_done));
  if (warp == 3) {
    if (lane == 0 && !mbar_wait(smem_u32(&s.roles_done), 0, nullptr, kWaitBudgetNs))
      report(prm.dev_status, MLA_ERR_DEVICE_TIMEOUT);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

}  // namespace tp

// ---------------------------------------------------------------------------- host

int tp_max_heads() { return 32; }

// Split ranges of the few-head kernel: one per SM.
int tp_max_ranges() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  if (cached[dev] > 0) return cached[dev];
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  cached[dev] = sms > 0 ? sms : 1;
  return cached[dev];
}

namespace {
// Encoded tensor maps, cached by address and shape (see decode_tc.cu).
struct TpKvEntry {
  bool valid;
  int dev;
  const void *base;
  int64_t rows;
  int32_t block_size;
  CUtensorMap kv4, kv1, kv2d;
};
struct TpQEntry {
  bool valid;
  int dev;
  const void *base;
  int32_t rows, box_rows;
  CUtensorMap q;
};
constexpr int kTpMapCacheSize = 64;
std::mutex g_tp_map_mu;
TpKvEntry g_tp_kv[kTpMapCacheSize];
TpQEntry g_tp_q[kTpMapCacheSize];

bool tp_maps(int dev, const void *cache, int64_t rows, int32_t block_size, const void *q,
             int32_t q_rows, int32_t hp, tp::Maps *m) {
  std::lock_guard<std::mutex> lock(g_tp_map_mu);
  TpKvEntry &e = g_tp_kv[tmap::slot_of_ptr(cache, kTpMapCacheSize)];
  if (!(e.valid && e.dev == dev && e.base == cache && e.rows == rows &&
        e.block_size == block_size)) {
    const uint32_t box_rows = block_size < tp::kTile ? (uint32_t)block_size : (uint32_t)tp::kTile;
    e.valid = false;
    if (!tmap::encode_3d(&e.kv4, cache, rows, box_rows, 4) ||
        !tmap::encode_3d(&e.kv1, cache, rows, box_rows, 1) ||
        !tmap::encode_2d(&e.kv2d, cache, rows, box_rows))
      return false;
    e.valid = true;
    e.dev = dev;
    e.base = cache;
    e.rows = rows;
    e.block_size = block_size;
  }
  TpQEntry &f = g_tp_q[tmap::slot_of_ptr(q, kTpMapCacheSize)];
  if (!(f.valid && f.dev == dev && f.base == q && f.rows == q_rows && f.box_rows == hp)) {
    f.valid = false;
    if (!tmap::encode_3d(&f.q, q, q_rows, (uint32_t)hp, tp::kChunks)) return false;
    f.valid = true;
    f.dev = dev;
    f.base = q;
    f.rows = q_rows;
    f.box_rows = hp;
  }
  m->kv4 = e.kv4;
  m->kv1 = e.kv1;
  m->kv2d = e.kv2d;
  m->q = f.q;
  return true;
}

template <int kHP>
cudaError_t launch_tp(const tp::Maps &maps, const tp::Params &p, int grid, cudaStream_t stream) {
  static std::atomic<bool> done[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(tp::Smem<kHP>) + 1024;
  if (!(dev >= 0 && dev < 64 && done[dev].load(std::memory_order_acquire))) {
    e = cudaFuncSetAttribute(tp::decode_tp_kernel<kHP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) done[dev].store(true, std::memory_order_release);
  }
  tp::decode_tp_kernel<kHP><<<grid, tp::kThreads, smem, stream>>>(maps, p);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_decode_tp(const void *q, const void *cache, int64_t num_blocks,
                             int32_t block_size, const int32_t *block_table,
                             int32_t max_blocks_per_seq, int32_t batch, int32_t heads,
                             float softmax_scale, void *out, float *lse, void *ws,
                             int32_t max_ranges, int32_t *dev_status, cudaStream_t stream) {
  if (heads < 1 || heads > tp_max_heads()) return cudaErrorInvalidValue;
  const int hp = heads <= 16 ? 16 : 32;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  tp::Maps maps;
  if (!tp_maps(dev, cache, num_blocks * (int64_t)block_size, block_size, q, batch * heads, hp,
               &maps))
    return cudaErrorInvalidValue;
  tp::Params p;
  p.block_table = block_table;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.block_size = block_size;
  p.num_blocks = (int32_t)num_blocks;
  p.batch = batch;
  p.heads = heads;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.out = (__nv_bfloat16 *)out;
  p.lse = lse;
  p.ws = ws;
  p.max_ranges = max_ranges;
  p.dev_status = dev_status;
  return hp == 16 ? launch_tp<16>(maps, p, max_ranges, stream)
                  : launch_tp<32>(maps, p, max_ranges, stream);
}

}  // namespace mla
