// Tensor-core MLA decode for sm_103a (tcgen05 + TMA + mbarrier pipeline).
//
// What is computed: absorbed-form MLA decode over the shared latent.  Every
// head's score uses all 576 dims of each cached row (512 kv_c + 64 k_rope
// shared by all heads) and the output is the softmax-weighted sum of the
// 512-dim kv_c  [dp-attention-expert-parallel-mla-kv-replication
// (inferenceinterviews.com), "A strong answer"; MLA 的 TP 切分 (10100.com),
// sections 2.2 and 3.1; DP 与 DPA 的区别 (chengxuchu.com), v_head_dim =
// kv_lora_rank].  All 128 heads read the same row, so the step is a dense
// contraction: S = Q K^T is [128 x 576] x [576 x tokens] and O = P V is
// [128 x tokens] x [tokens x 512], run on the tensor cores (M = 128 heads).
//
// Layout of the work.  The fp32 output of one request, 128 heads x 512 dims,
// is exactly one SM's tensor memory, which would leave no room for S.  So two
// CTAs share a split range of the plan and split the OUTPUT dims: CTA r owns
// O[:, 256r .. 256r+255].  Each CTA computes the full score S itself (the QK
// contraction is done by both CTAs: moving partial scores between SMs costs
// more than recomputing them), then P V for its half.  Both CTAs read the same
// tiles at about the same time, so the second read is served by L2.
//
// Operands.  Q's 256 "own" kv_c dims live in tensor memory (A operand: staged
// in shared memory by TMA at each segment start and copied over with
// tcgen05.cp); its other 256 dims and its 64 rope dims live in shared memory
// (A operand from a shared-memory descriptor).  S is double-buffered in tensor memory, so the S
// MMAs of the next tile run while the softmax works on this one; P (bf16) is
// written over the S buffer it came from and read from there by P V.  A 64-token cache tile arrives by TMA in two large boxes,
// 128-byte swizzled: the "other" part (the other 256 kv_c dims + 64 rope dims)
// and the "own" part (this CTA's 256 value dims).  S is accumulated over the
// other dims first, then rope, then the own dims, so the other part of a slot
// is released early and refilled 1.5 tiles ahead, while the own part (also the
// V operand of P V) is held until P V and is needed only at the end of the
// next-but-one S: two slots per part hide the load latency.  (L2 prefetch of
// upcoming tiles, whole or only their other part, measured slower here: it
// adds TMA instructions on the producer's critical path and, at launch, a
// burst that delays every CTA's first tiles.)
//
// Warp roles: warp 0 loads the own parts; warp 3 loads the other parts;
// warp 9 loads every segment's Q; warps 1 and 8 issue
// the S MMAs of even and odd tiles; warp 2 issues the P V MMAs;
// warps 4-7 (one thread per head) run the online softmax with lazy rescaling
// of O and write the output (or split partials plus log-sum-exp); warp 4 owns
// the tensor memory allocation.
//
// Launch order.  Launched as a programmatic dependent of the previous kernel
// (early_launch), a CTA sets up its barriers and tensor memory while that
// kernel ends and, before griddepcontrol.wait, only asks L2 for its first
// tile and q; everything it reads or writes comes after the wait.  Each CTA
// releases its own dependents once it has requested its last tile.
//
// FP8 cache (kFp8).  The cache holds one E4M3 byte per element, 576 bytes per
// token per layer [MLA 的 TP 切分 (10100.com), opening paragraph and section
// 5.1], with one scale per layer (a code c stands for value(c) * kv_scale).
// Each part of a tile lands by TMA in the upper half of its 16-bit slot and
// two more warps (10: the other part, 11: the own part) widen it in place to
// f16, which holds every E4M3 value exactly; the MMAs then run on f16
// operands (kind::f16 needs A and B of one type), so each segment's q is also
// turned into f16 in place once it lands (exact for |q| in [2^-14, 65504],
// saturating above), and P is packed as f16.  kv_scale leaves the MMAs: the
// scores use softmax_scale * kv_scale, the output is multiplied by kv_scale.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "fp8.cuh"
#include "sm100.cuh"
#include "tmap.h"

namespace mla {
namespace tc {

using namespace sm100;

constexpr int kTile = 64;                  // tokens per tile (= plan unit)
constexpr int kSlots = 2;                  // slots per part
constexpr int kVHalf = 256;                // output dims per CTA
constexpr int kChunkBytes = kTile * 128;   // one 64-dim, 64-token SW128 chunk: 8 KB
constexpr int kQChunkBytes = 128 * 128;    // one 64-dim chunk of Q for 128 heads: 16 KB
constexpr int kThreads = 320;              // 10 warps (bf16 cache)
constexpr int kThreadsFp8 = 384;           // 12 warps: + two FP8 converter warps
constexpr int kOtherStage = 20 * 1024;     // FP8 staging: upper half of an "other" slot
constexpr int kOwnStage = 16 * 1024;       // FP8 staging: upper half of an "own" slot
constexpr int kChunkBytes8 = kTile * 64;   // one 64-dim, 64-token FP8 chunk: 4 KB
constexpr int kSoftmaxThreads = 128;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 256, kColQ = 384;  // S buffers at kColS + 64 * (g & 1)
constexpr uint64_t kWaitBudgetNs = 100000000ull;  // 100 ms per wait, far above any legal wait
constexpr uint64_t kDrainBudgetNs = 10000000ull;  // 10 ms to drain in-flight copies on abort
constexpr float kRescaleThreshold = 8.0f;         // log2 units

struct __align__(1024) Smem {
  uint8_t q_other[4][kQChunkBytes];      // Q[:, other 256 dims], 4 chunks of 64 dims: 64 KB
                                         // (at a segment start: Q[:, own dims], staged)
  uint8_t q_rope[kQChunkBytes];          // Q[:, 64 rope dims]: 16 KB
  uint8_t other[kSlots][5][kChunkBytes]; // other 256 kv_c dims (4 chunks) + rope: 40 KB / slot
  uint8_t own[kSlots][4][kChunkBytes];   // own 256 value dims: 32 KB / slot
  uint64_t other_full[kSlots], other_empty[kSlots], own_full[kSlots], own_empty[kSlots];
  // per S buffer: S ready / P written over it / P V of that buffer's tile done.
  // P has one barrier per buffer: the softmax warps run independently, and a
  // warp may already write the next tile's P while another is still on this
  // one; a single 128-arrival barrier would then count arrivals of two tiles
  // in one phase.  No warp gets two tiles ahead (S of tile g+2 waits for the
  // P V of tile g), so two barriers suffice.
  uint64_t s_full[2], p_full[2], pv_done[2];
  // S MMAs of tile g all issued: the two S issuers take turns tile by tile, so
  // the pipe finishes one tile's S before the next (its softmax, P V and the
  // S-buffer reuse two tiles on depend on it) instead of interleaving both.
  uint64_t qk_seq[2];
  uint64_t qown_full, q_full, q_tmem, q_free, fin_qk, fin_pv, row_ready;
  uint64_t stage_free;  // one phase: the staged first Q own dims have been copied
  // FP8 cache: the TMA of a part landed in its staging half (other/own), and
  // each segment's q was turned into f16 (own dims + rope / other dims)
  uint64_t other_staged[kSlots], own_staged[kSlots], qown_conv, q_conv;
  // one phase: every warp is done with its role (all its tensor-memory work,
  // the operations it issued complete)
  uint64_t roles_done;
  uint32_t tmem_base;
  int abort;
};

// At launch the first segment's Q own dims (four 16 KB chunks) are staged in
// slot 1 of both rings, which stay empty until tile 1: chunks 0-1 in the
// other ring's slot 1, chunks 2-3 in the own ring's slot 1.  Tile 0's loads
// then need not wait for the copy into tensor memory.
__device__ __forceinline__ uint8_t *q_stage_chunk(Smem &s, int c) {
  return c < 2 ? s.other[1][2 * c] : s.own[1][2 * (c - 2)];
}
static_assert(2 * kChunkBytes == kQChunkBytes, "a Q chunk is two cache chunks");

// Tensor maps over the cache viewed as [rows = NB*BS][576]: 3-D views
// {64 columns, rows, 9 chunks} (chunk stride 128 B) fetch several 64-dim
// chunks of 64 rows in one box, laid out chunk after chunk; the 2-D view
// serves pages shorter than a tile.
struct Maps {
  CUtensorMap kv5, kv4, kv1, kv2d, q;
};

struct Params {
  const __nv_bfloat16 *q;
  const int32_t *block_table;
  int32_t max_blocks_per_seq;
  int32_t block_size;
  int32_t num_blocks;
  int32_t batch;
  float scale_log2;
  __nv_bfloat16 *out;
  float *lse;
  void *ws;
  int32_t max_ranges;
  int32_t *dev_status;
  const uint4 *kv_new;  // optional: row b is request b's newest token, stored before decoding
  uint4 *cache_rows;    // the cache, for those stores
  float kv_scale;       // FP8 cache: the value of a code is value(code) * kv_scale
  float kv_inv_scale;   // FP8 cache: a new row is stored as code(x * kv_inv_scale)
  int32_t early_launch; // launched as a programmatic dependent (see griddep_wait below)
};

__device__ __forceinline__ void set_abort(Smem &s, int32_t *dev_status) {
  s.abort = 1;
  report(dev_status, MLA_ERR_DEVICE_TIMEOUT);
}

// Every lane polls (each gets the barrier's acquire), then the warp agrees, so
// control flow around warp-collective tcgen05 instructions stays uniform.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const volatile int *abort) {
  const bool ok = mbar_wait(bar, parity, abort, kWaitBudgetNs);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// FP8 cache: widen one part of a tile (nch chunks of 64 dims x 64 rows) from
// its E4M3 staging (chunk c at stage + 4 KB c, row r at + 64 r) to f16 in the
// 128-byte-swizzled operand layout (chunk c at dst + 8 KB c, row r at + 128 r,
// 16-byte unit u at ((u ^ (r & 7)) << 4)).  One warp, a chunk at a time: lane
// l reads 16 staging bytes of rows l/4, l/4 + 8, ..., all eight loads in
// flight, converts them, and writes them only after the whole warp has read
// the chunk.  The staging is the upper half of the same slot; a chunk's
// writes end at or before the first staging byte of the next chunk (for
// every chunk of either part: 8 KB (c + 1) <= stage offset + 4 KB (c + 1)).
template <int kNch>
__device__ __forceinline__ void widen_part_fp8(uint8_t *dst, const uint8_t *stage, int lane) {
  const int q4 = lane & 3, r0 = lane >> 2;
#pragma unroll 1
  for (int c = 0; c < kNch; ++c) {
    uint4 v[kTile / 8];
#pragma unroll
    for (int it = 0; it < kTile / 8; ++it)
      v[it] = *reinterpret_cast<const uint4 *>(stage + c * kChunkBytes8 + (it * 8 + r0) * 64 +
                                               q4 * 16);
    __syncwarp();  // the whole chunk is read before any of it is overwritten
#pragma unroll
    for (int it = 0; it < kTile / 8; ++it) {
      const int r = it * 8 + r0;
      uint4 o0, o1;
      o0.x = e4m3x2_to_f16x2(v[it].x); o0.y = e4m3x2_to_f16x2(v[it].x >> 16);
      o0.z = e4m3x2_to_f16x2(v[it].y); o0.w = e4m3x2_to_f16x2(v[it].y >> 16);
      o1.x = e4m3x2_to_f16x2(v[it].z); o1.y = e4m3x2_to_f16x2(v[it].z >> 16);
      o1.z = e4m3x2_to_f16x2(v[it].w); o1.w = e4m3x2_to_f16x2(v[it].w >> 16);
      uint8_t *row = dst + c * kChunkBytes + r * 128;
      *reinterpret_cast<uint4 *>(row + (((2 * q4) ^ (r & 7)) << 4)) = o0;
      *reinterpret_cast<uint4 *>(row + (((2 * q4 + 1) ^ (r & 7)) << 4)) = o1;
    }
    __syncwarp();
  }
}

// FP8 cache: turn bytes of bf16 q in shared memory into f16 in place (the
// operand layout is the same for both 16-bit types).  One warp, eight 16-byte
// words per lane in flight.
__device__ __forceinline__ void q_to_f16(uint8_t *buf, int bytes, int lane) {
  constexpr int kStep = 32 * 16 * 8;
  for (int base = 0; base < bytes; base += kStep) {
    uint4 w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      w[k] = *reinterpret_cast<const uint4 *>(buf + base + (k * 32 + lane) * 16);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      w[k].x = bf16x2_to_f16x2(w[k].x); w[k].y = bf16x2_to_f16x2(w[k].y);
      w[k].z = bf16x2_to_f16x2(w[k].z); w[k].w = bf16x2_to_f16x2(w[k].w);
      *reinterpret_cast<uint4 *>(buf + base + (k * 32 + lane) * 16) = w[k];
    }
  }
}

template <bool kFp8>
__global__ void __launch_bounds__(kFp8 ? kThreadsFp8 : kThreads, 1)
    decode_tc_kernel(const __grid_constant__ Maps maps, const Params prm) {
  constexpr int kNumThreads = kFp8 ? kThreadsFp8 : kThreads;
  extern __shared__ uint8_t smem_raw[];
  Smem &s = *reinterpret_cast<Smem *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int half = blockIdx.x & 1;  // this CTA owns output dims [256*half, 256*half + 256)
  const int pair = blockIdx.x >> 1;
  const PlanView v = plan_view(prm.ws, prm.batch, kHeads, prm.max_ranges);
  const volatile int *abort_flag = &s.abort;
  // This range's segment count and first segment record, requested before
  // the setup below so that their latency overlaps it; launched early, only
  // their lines are fetched into L2 now, and they are read once the previous
  // kernel has completed (griddep_wait below).
  int32_t seg_n = 0;
  SegRec seg_first = {};
  if (!prm.early_launch) {
    seg_n = v.seg_count[pair];
    seg_first = v.seg_rec[(int64_t)pair * kSegCache];
  } else if (tid == 32) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(v.seg_count + pair) : "memory");
    asm volatile("prefetch.global.L2 [%0];" ::"l"(v.seg_rec + (int64_t)pair * kSegCache) : "memory");
  }

  if (tid == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(smem_u32(&s.other_full[i]), 1);
      mbar_init(smem_u32(&s.other_empty[i]), 1);
      mbar_init(smem_u32(&s.own_full[i]), 1);
      mbar_init(smem_u32(&s.own_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s.s_full[i]), 1);
      mbar_init(smem_u32(&s.p_full[i]), kSoftmaxThreads);
      mbar_init(smem_u32(&s.pv_done[i]), 1);
      mbar_init(smem_u32(&s.qk_seq[i]), 1);
    }
    mbar_init(smem_u32(&s.qown_full), 1);
    mbar_init(smem_u32(&s.row_ready), 1);
    mbar_init(smem_u32(&s.stage_free), 1);
    mbar_init(smem_u32(&s.q_full), 1);
    mbar_init(smem_u32(&s.q_tmem), 1);  // tcgen05.commit of the Q-own copy
    mbar_init(smem_u32(&s.q_free), 2);  // both S issuers
    mbar_init(smem_u32(&s.fin_qk), 2);
    mbar_init(smem_u32(&s.fin_pv), 1);
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(smem_u32(&s.other_staged[i]), 1);
      mbar_init(smem_u32(&s.own_staged[i]), 1);
    }
    mbar_init(smem_u32(&s.qown_conv), 1);
    mbar_init(smem_u32(&s.q_conv), 1);
    mbar_init(smem_u32(&s.roles_done), kNumThreads / 32);
    s.abort = 0;
    fence_mbarrier_init_cluster();
  }
  if (warp == 4) {  // a softmax warp: among the last to finish, it also frees it
    tmem_alloc(smem_u32(&s.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  __syncwarp();  // warps reach the CTA barrier converged (thread 0 alone did the setup)
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  // Launched as a programmatic dependent (after a one-wave combine), the
  // setup above ran during the previous kernel's tail; everything below —
  // the plan, q, the cache, the outputs, the partials — waits for it to
  // complete and for its writes to be visible.
  if (!kFp8 && prm.early_launch && (warp == 0 || warp == 3 || warp == 9) && lane == 0) {
    // While the previous kernel ends: the first tile's parts and the first
    // request's q towards L2, at the places the plan's first record names.
    // Read before the wait, that record may be stale: it only aims these
    // prefetches (out-of-range boxes fetch nothing), and everything is read
    // again after the wait.
    const int32_t n0 = v.seg_count[pair];
    const SegRec r0 = v.seg_rec[(int64_t)pair * kSegCache];
    if (n0 <= 0 || r0.b < 0 || r0.b >= prm.batch) {
      // nothing to aim at
    } else if (warp == 9) {
      for (int c = 0; c < kRow / 64; ++c) tma_prefetch_2d(&maps.q, 64 * c, r0.b * kHeads);
    } else if (r0.row0 >= 0 && prm.block_size >= kTile) {
      if (warp == 0) {
        tma_prefetch_3d(&maps.kv4, 0, r0.row0, half * 4);
      } else if (half == 0) {
        tma_prefetch_3d(&maps.kv5, 0, r0.row0, 4);
      } else {
        tma_prefetch_3d(&maps.kv4, 0, r0.row0, 0);
        tma_prefetch_3d(&maps.kv1, 0, r0.row0, 8);
      }
    }
  }
  griddep_wait();
  if (prm.early_launch) {
    seg_n = v.seg_count[pair];
    seg_first = v.seg_rec[(int64_t)pair * kSegCache];
  }

  const bool active = seg_n > 0;  // ranges past the plan's count have none
  // Whether the plan was made for these arguments (see plan_record_ok).  Only
  // the roles that form global addresses from the plan's records check it,
  // each at its first record (where it waits for that record anyway): the
  // producers (block-table reads), the appended rows and the softmax
  // (output writes).  A producer that finds a plan made for other arguments
  // reports it and raises the abort flag, which ends the other roles.
  const int32_t seg_stamp =
      plan_stamp(prm.batch, prm.max_ranges, kTile, prm.block_size, prm.max_blocks_per_seq);
  auto plan_ok = [&]() {
    return plan_record_ok(seg_n, seg_first, seg_stamp, prm.batch,
                          prm.max_blocks_per_seq * prm.block_size, 2 * prm.max_ranges);
  };
  const int own0 = half * 4;        // first own 64-dim chunk (of the 8 kv_c chunks)
  const int oth0 = (1 - half) * 4;  // first other chunk
  const int BS = prm.block_size;
  const bool big_pages = BS >= kTile;  // a tile lies inside one page: one box per part

  if (warp == 0 || warp == 3) {
    // ------------------------------------------------------------ TMA producers
    if (active && elect_one_sync()) {
      const bool own_role = (warp == 0);
      // the plan's records address the block table: a plan made for other
      // arguments stops both producers here, and the abort flag the others
      const bool plan_good = plan_ok();
      if (!plan_good) {
        s.abort = 1;
        report(prm.dev_status, MLA_ERR_DEVICE_PLAN);
      }
      // normal priority: the pair's other CTA reads every tile too, usually a
      // little later; evict-first lines were often gone by then (ncu: ~19%
      // extra DRAM reads on a 64 x 4096 layer)
      const uint64_t policy = policy_evict_normal();
      SegIter<kTile> it;
      it.init(v, prm.batch, pair, seg_n, seg_first);
      int32_t t0, t1, slot_p;
      uint32_t g = 0;
      const int box_rows = BS < kTile ? BS : kTile;
      const uint32_t box_bytes = (uint32_t)(box_rows * (kFp8 ? 64 : 128));
      // where chunk c, page box j of a part lands: its 16-bit slot, or with an
      // FP8 cache the staging half of that slot
      auto part_dst = [&](const uint8_t *slot_base, int stage_off, int c, int j) -> uint32_t {
        return kFp8 ? smem_u32(slot_base) + stage_off + c * kChunkBytes8 + j * box_bytes
                    : smem_u32(slot_base) + c * kChunkBytes + j * box_bytes;
      };
      const int64_t nb = prm.num_blocks;
      // Block-table entries of the next tile are loaded one tile ahead into
      // registers: plain loads whose latency overlaps this tile's slot wait.
      // A segment's first tile needs none when the plan's record has its row.
      SegIter<kTile> fc = it;  // shares the first record load
      int32_t fc_t = 0, fc_t1 = 0, fc_slot;
      bool fc_more = true;
      int32_t nxt[kTile / 16];
      auto load_next = [&]() {  // move the cursor one tile on and load that tile's entries
        bool first = false;
        while (fc_more && fc_t >= fc_t1) {
          fc_more = fc.next(fc_t, fc_t1, fc_slot);
          first = true;
        }
        if (!fc_more) return;
        if (!(first && fc.row0 >= 0 && big_pages)) {
          const int32_t *row = prm.block_table + (int64_t)fc.b * prm.max_blocks_per_seq;
          const int nbx = (min(kTile, fc_t1 - fc_t) + box_rows - 1) / box_rows;
#pragma unroll
          for (int j = 0; j < kTile / 16; ++j)
            if (j < nbx) nxt[j] = row[(fc_t + j * box_rows) / BS];
        }
        fc_t += kTile;
      };
      if (plan_good) load_next();
      if (own_role) {
        prefetch_tmap(&maps.kv4);
      } else {
        prefetch_tmap(&maps.kv5);
        prefetch_tmap(&maps.kv1);
      }
      bool ok = plan_good;
      while (ok && it.next(t0, t1, slot_p)) {
        for (int32_t tt = t0; tt < t1; tt += kTile, ++g) {
          // cache rows of the tile's boxes (one box per page, or one per tile):
          // a segment's first tile from the plan's record when it has one,
          // else from the entries loaded one tile ago
          const int nbx = (min(kTile, t1 - tt) + box_rows - 1) / box_rows;
          int32_t y[kTile / 16];
          if (tt == t0 && it.row0 >= 0 && big_pages) {
            y[0] = it.row0;
          } else {
#pragma unroll
            for (int j = 0; j < kTile / 16; ++j) {
              if (j >= nbx) break;
              int32_t blk = nxt[j];
              if (blk < 0 || blk >= nb) {
                if (own_role) report(prm.dev_status, MLA_ERR_DEVICE_RANGE);
                blk = 0;
              }
              y[j] = blk * BS + ((tt + j * box_rows) % BS);
            }
          }
          load_next();  // the next tile's entries, consumed one iteration later
          const int slot = g % kSlots;
          const uint32_t par = ((g / kSlots) & 1u) ^ 1u;
          // the tile holding a request's newest row, when this launch stores it
          if (prm.kv_new && tt + kTile >= t1 && t1 == v.seq_len[it.b] &&
              !mbar_wait(smem_u32(&s.row_ready), 0, abort_flag, kWaitBudgetNs)) {
            set_abort(s, prm.dev_status);
            ok = false;
            break;
          }
          if (own_role) {
            // slot 1 stages the first segment's Q own dims until they have
            // been copied to tensor memory
            if (g == 1 && !mbar_wait(smem_u32(&s.stage_free), 0, abort_flag, kWaitBudgetNs)) {
              set_abort(s, prm.dev_status);
              ok = false;
              break;
            }
            if (!mbar_wait(smem_u32(&s.own_empty[slot]), par, abort_flag, kWaitBudgetNs)) {
              set_abort(s, prm.dev_status);
              ok = false;
              break;
            }
            const uint32_t bar = smem_u32(kFp8 ? &s.own_staged[slot] : &s.own_full[slot]);
            mbar_arrive_expect_tx(bar, 4u * nbx * box_bytes);
            if (big_pages) {
              tma_load_3d_hint(part_dst(s.own[slot][0], kOwnStage, 0, 0), &maps.kv4, 0, y[0], own0,
                               bar, policy);
            } else {
#pragma unroll
              for (int j = 0; j < kTile / 16; ++j) {
                if (j >= nbx) break;
                for (int c = 0; c < 4; ++c)
                  tma_load_2d_hint(part_dst(s.own[slot][0], kOwnStage, c, j), &maps.kv2d,
                                   64 * (own0 + c), y[j], bar, policy);
              }
            }
          } else {
            if (g == 1 && !mbar_wait(smem_u32(&s.stage_free), 0, abort_flag, kWaitBudgetNs)) {
              set_abort(s, prm.dev_status);
              ok = false;
              break;
            }
            if (!mbar_wait(smem_u32(&s.other_empty[slot]), par, abort_flag, kWaitBudgetNs)) {
              set_abort(s, prm.dev_status);
              ok = false;
              break;
            }
            const uint32_t bar = smem_u32(kFp8 ? &s.other_staged[slot] : &s.other_full[slot]);
            mbar_arrive_expect_tx(bar, 5u * nbx * box_bytes);
            if (big_pages) {
              if (half == 0) {  // other = chunks 4..7, rope = chunk 8: contiguous
                tma_load_3d_hint(part_dst(s.other[slot][0], kOtherStage, 0, 0), &maps.kv5, 0, y[0],
                                 4, bar, policy);
              } else {          // other = chunks 0..3, then rope
                tma_load_3d_hint(part_dst(s.other[slot][0], kOtherStage, 0, 0), &maps.kv4, 0, y[0],
                                 0, bar, policy);
                tma_load_3d_hint(part_dst(s.other[slot][0], kOtherStage, 4, 0), &maps.kv1, 0, y[0],
                                 8, bar, policy);
              }
            } else {
#pragma unroll
              for (int j = 0; j < kTile / 16; ++j) {
                if (j >= nbx) break;
                for (int c = 0; c < 5; ++c)
                  tma_load_2d_hint(part_dst(s.other[slot][0], kOtherStage, c, j), &maps.kv2d,
                                   c < 4 ? 64 * (oth0 + c) : 512, y[j], bar, policy);
              }
            }
          }
        }
      }
      // every tile requested: a split combine launched as a programmatic
      // dependent may start its blocks on SMs this grid frees (it waits for
      // the whole grid before it reads anything)
      if (own_role) griddep_launch_dependents();
      if (s.abort && plan_good) {
        // the consumers gave up: let the last issued loads land before exit
        for (int i = 0; i < kSlots; ++i) {
          uint64_t *landed = kFp8 ? (own_role ? &s.own_staged[i] : &s.other_staged[i])
                                  : (own_role ? &s.own_full[i] : &s.other_full[i]);
          (void)mbar_wait(smem_u32(landed), 0, nullptr, kDrainBudgetNs);
        }
      }
    }
  } else if (warp == 1 || warp == 8) {
    // ------------------------------------------------------------ S = Q K^T issuers
    // Warp 1 issues the S MMAs of even tiles, warp 8 those of odd tiles: one
    // thread cannot issue N = 64 MMAs as fast as the tensor pipe runs them.
    // They take turns (qk_seq), one whole tile each.
    // Tile g uses S buffer g & 1 and ring slot g % 2, so the two never touch
    // the same accumulator or operands.  Both wait for every segment's Q and
    // both release it (q_free counts two arrivals); the even issuer also
    // copies the segment's Q own dims into tensor memory.
    const uint32_t par = warp == 8 ? 1u : 0u;
    if (active && elect_one_sync()) {
      SegIter<kTile> it;
      it.init(v, prm.batch, pair, seg_n, seg_first);
      int32_t t0, t1, slot_p;
      uint32_t g = 0, seg = 0;
      const uint32_t id = kFp8 ? idesc_f16_f32(128, kTile, 0) : idesc_bf16_f32(128, kTile, 0);
      // Q in place: its TMA with a bf16 cache, its conversion to f16 with FP8
      uint64_t *qown_ready = kFp8 ? &s.qown_conv : &s.qown_full;
      uint64_t *qoth_ready = kFp8 ? &s.q_conv : &s.q_full;
      // descriptors of slot 0 / chunk 0; chunks, slots and k-steps add their
      // byte offset >> 4 to the 14-bit start-address field (no carry: every
      // shared-memory address here is below 2^18)
      const uint64_t d_own = smem_desc(smem_u32(s.own[0][0]), 16, 1024, kSwizzle128B);
      const uint64_t d_oth = smem_desc(smem_u32(s.other[0][0]), 16, 1024, kSwizzle128B);
      const uint64_t d_q = smem_desc(smem_u32(s.q_other[0]), 16, 1024, kSwizzle128B);
      const uint64_t d_rope = smem_desc(smem_u32(s.q_rope), 16, 1024, kSwizzle128B);
      const uint32_t a_q = tmem + kColQ;
      bool ok = true;
      while (ok && it.next(t0, t1, slot_p)) {
        if (!mbar_wait(smem_u32(qown_ready), seg & 1u, abort_flag, kWaitBudgetNs)) {
          set_abort(s, prm.dev_status);
          break;
        }
        if (par == 0) {
          // Q[:, own 256 dims] into tensor memory: 16 copies of 128 rows x 16
          // dims, addressed like the A operand.  Staged in the rings' slot 1
          // for the first segment, in the Q buffers afterwards.
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint64_t d_src =
                seg == 0 ? smem_desc(smem_u32(q_stage_chunk(s, c)), 16, 1024, kSwizzle128B)
                         : d_q + (uint64_t)((c * kQChunkBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tmem_cp_128x256b(a_q + c * 32 + kk * 8, d_src + (uint64_t)((kk * 32) >> 4));
          }
          mma_commit(smem_u32(&s.q_tmem));
          if (seg == 0) mma_commit(smem_u32(&s.stage_free));
        }
        if (!mbar_wait(smem_u32(&s.q_tmem), seg & 1u, abort_flag, kWaitBudgetNs) ||
            !mbar_wait(smem_u32(qoth_ready), seg & 1u, abort_flag, kWaitBudgetNs)) {
          set_abort(s, prm.dev_status);
          break;
        }
        ++seg;
        tc_fence_after();
        for (int32_t tt = t0; tt < t1; tt += kTile, ++g) {
          if ((g & 1u) != par) continue;  // the other issuer's tile
          const int slot = g % kSlots;
          const uint32_t ph = (g / kSlots) & 1u;
          const uint32_t d_s = tmem + kColS + 64 * (g & 1u);
          if (g >= 1 && !mbar_wait(smem_u32(&s.qk_seq[(g - 1) & 1u]), ((g - 1) >> 1) & 1u,
                                   abort_flag, kWaitBudgetNs)) {
            set_abort(s, prm.dev_status);
            ok = false;
            break;
          }
          // The S buffer is overwritten only once the P V of tile g-2, which
          // reads P from it, has completed.  Issued is not enough: MMAs issued
          // by different threads are not run in issue order (with only the
          // issue ordered, through a barrier and the tcgen05 fences around it,
          // P V read S values in place of P, a few heads per tile in ~97% of
          // runs of a 64 x 4096 layer).
          if (!mbar_wait(smem_u32(&s.other_full[slot]), ph, abort_flag, kWaitBudgetNs) ||
              (g >= 2 && !mbar_wait(smem_u32(&s.pv_done[g & 1u]), ((g >> 1) - 1) & 1u,
                                    abort_flag, kWaitBudgetNs))) {
            set_abort(s, prm.dev_status);
            ok = false;
            break;
          }
          tc_fence_after();
          // other 256 kv_c dims, then rope: A = Q (shared memory), B = other part
          const uint64_t bo = d_oth + (uint64_t)((slot * 5 * kChunkBytes) >> 4);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t a = d_q + (uint64_t)((c * kQChunkBytes + kk * 32) >> 4);
              const uint64_t b = bo + (uint64_t)((c * kChunkBytes + kk * 32) >> 4);
              if (c == 0 && kk == 0) mma_ss(d_s, a, b, id, 0); else mma_ss_acc(d_s, a, b, id);
            }
          }
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss_acc(d_s, d_rope + (uint64_t)((kk * 32) >> 4),
                       bo + (uint64_t)((4 * kChunkBytes + kk * 32) >> 4), id);
          mma_commit(smem_u32(&s.other_empty[slot]));
          // own 256 kv_c dims: A = Q (tensor memory), B = own part
          if (!mbar_wait(smem_u32(&s.own_full[slot]), ph, abort_flag, kWaitBudgetNs)) {
            set_abort(s, prm.dev_status);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bw = d_own + (uint64_t)((slot * 4 * kChunkBytes) >> 4);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ts_acc(d_s, a_q + c * 32 + kk * 8,
                         bw + (uint64_t)((c * kChunkBytes + kk * 32) >> 4), id);
          }
          mma_commit(smem_u32(&s.s_full[g & 1u]));
          mbar_arrive(smem_u32(&s.qk_seq[g & 1u]));
        }
        if (!ok) break;
        mma_commit(smem_u32(&s.q_free));  // Q of this segment no longer read
      }
      mma_commit(smem_u32(&s.fin_qk));
      if (!mbar_wait(smem_u32(&s.fin_qk), 0, nullptr, kWaitBudgetNs))
        report(prm.dev_status, MLA_ERR_DEVICE_TIMEOUT);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ O += P V issuer
    if (active && elect_one_sync()) {
      SegIter<kTile> it;
      it.init(v, prm.batch, pair, seg_n, seg_first);
      int32_t t0, t1, slot_p;
      uint32_t g = 0;
      const uint32_t id_pv = kFp8 ? idesc_f16_f32(128, kVHalf, 1) : idesc_bf16_f32(128, kVHalf, 1);
      const uint64_t d_own = smem_desc(smem_u32(s.own[0][0]), kChunkBytes, 1024, kSwizzle128B);
      bool ok = true;
      while (ok && it.next(t0, t1, slot_p)) {
        for (int32_t tt = t0; tt < t1; tt += kTile, ++g) {
          const int n = min(kTile, t1 - tt);
          const int slot = g % kSlots;
          if (!mbar_wait(smem_u32(&s.p_full[g & 1u]), (g >> 1) & 1u, abort_flag, kWaitBudgetNs)) {
            set_abort(s, prm.dev_status);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bw = d_own + (uint64_t)((slot * 4 * kChunkBytes) >> 4);
          const uint32_t a_p = tmem + kColS + 64 * (g & 1u);  // P sits in its S buffer
          const int ksteps = (n + 15) >> 4;
          for (int kt = 0; kt < ksteps; ++kt)
            mma_ts(tmem + kColO, a_p + kt * 8, bw + (uint64_t)((kt * 2048) >> 4), id_pv,
                   (tt > t0 || kt > 0) ? 1u : 0u);
          mma_commit(smem_u32(&s.pv_done[g & 1u]));
          mma_commit(smem_u32(&s.own_empty[slot]));
        }
      }
      mma_commit(smem_u32(&s.fin_pv));
      if (!mbar_wait(smem_u32(&s.fin_pv), 0, nullptr, kWaitBudgetNs))
        report(prm.dev_status, MLA_ERR_DEVICE_TIMEOUT);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ Q loader and appended rows
    // Q of every segment's request, once the previous segment's S MMAs are
    // done with the Q buffers: first its own 256 dims (and rope), from where
    // the even S issuer copies the own dims into tensor memory (tcgen05.cp),
    // then, once copied, its other 256 dims.  A warp of its own, so that the
    // tile loads never wait behind Q.
    //
    // With kv_new, request b's newest row (token seq_len[b] - 1) is stored
    // into its slot by the CTAs whose range holds that token, before their
    // producers load the tile holding it: the warp writes the rows, orders
    // them before the async proxy's reads, and signals row_ready.  Both CTAs
    // of the pair store the same bytes, each before its own loads.  The first
    // segment's Q goes out before these stores, whose table lookups are
    // dependent loads: the first S MMAs need Q, while the newest row is
    // usually needed tiles later.
    if (active) {
      const bool leader = elect_one_sync();
      SegIter<kTile> qi;
      qi.init(v, prm.batch, pair, seg_n, seg_first);
      int32_t qt0, qt1, qslot;
      uint32_t seg = 0;
      bool qok = true;
      // one segment's Q loads; false when a wait gave up
      auto load_q = [&]() -> bool {
        if (!mbar_wait(smem_u32(&s.q_free), (seg & 1u) ^ 1u, abort_flag, kWaitBudgetNs)) {
          set_abort(s, prm.dev_status);
          return false;
        }
        // own dims: into the rings' slot 1 for the first segment (empty until
        // the copy is done, so Q's other dims need not wait), else the Q buffers
        mbar_arrive_expect_tx(smem_u32(&s.qown_full), 5 * kQChunkBytes);
        for (int c = 0; c < 4; ++c)
          tma_load_2d(smem_u32(seg == 0 ? q_stage_chunk(s, c) : s.q_other[c]), &maps.q,
                      64 * (own0 + c), qi.b * kHeads, smem_u32(&s.qown_full));
        tma_load_2d(smem_u32(s.q_rope), &maps.q, 512, qi.b * kHeads, smem_u32(&s.qown_full));
        {  // the next segment's Q rows into L2 meanwhile
          SegIter<kTile> nx = qi;
          int32_t a0, a1, aslot;
          if (nx.next(a0, a1, aslot))
            for (int c = 0; c < 9; ++c) tma_prefetch_2d(&maps.q, 64 * c, nx.b * kHeads);
        }
        if (seg > 0 && !mbar_wait(smem_u32(&s.q_tmem), seg & 1u, abort_flag, kWaitBudgetNs)) {
          set_abort(s, prm.dev_status);
          return false;
        }
        mbar_arrive_expect_tx(smem_u32(&s.q_full), 4 * kQChunkBytes);
        for (int c = 0; c < 4; ++c)
          tma_load_2d(smem_u32(s.q_other[c]), &maps.q, 64 * (oth0 + c), qi.b * kHeads,
                      smem_u32(&s.q_full));
        ++seg;
        return true;
      };
      // the first segment's Q (its waits pass at once)
      if (leader && qi.next(qt0, qt1, qslot)) qok = load_q();
      __syncwarp();
      if (prm.kv_new && plan_ok()) {  // the rows' slots come from the plan's records
        SegIter<kTile> it;
        it.init(v, prm.batch, pair, seg_n, seg_first);
        int32_t t0, t1, slot_p;
        while (it.next(t0, t1, slot_p)) {
          const int32_t L = v.seq_len[it.b];
          if (t1 != L || L == 0) continue;  // not the request's last segment
          const int32_t pos = L - 1;
          const int32_t blk = prm.block_table[(int64_t)it.b * prm.max_blocks_per_seq + pos / BS];
          if (blk < 0 || blk >= prm.num_blocks) {
            if (lane == 0) report(prm.dev_status, MLA_ERR_DEVICE_RANGE);
            continue;
          }
          const int64_t row = (int64_t)blk * BS + pos % BS;
          const uint4 *src = prm.kv_new + (int64_t)it.b * (kRow / 8);
          if (kFp8) {  // 8 elements (16 bytes of bf16) -> 8 codes per word
            uint2 *dst = reinterpret_cast<uint2 *>(prm.cache_rows) + row * (kRow / 8);
            for (int k = lane; k < kRow / 8; k += 32)
              dst[k] = quantize_bf16x8(__ldg(src + k), prm.kv_inv_scale);
          } else {
            uint4 *dst = prm.cache_rows + row * (kRow / 8);
            for (int k = lane; k < kRow / 8; k += 32) dst[k] = __ldg(src + k);
          }
        }
        fence_proxy_async_global();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s.row_ready));
      }
      if (leader) {
        // later segments' Q, each after the previous segment's S MMAs
        while (qok && qi.next(qt0, qt1, qslot)) qok = load_q();
        if (s.abort) {  // let the last issued loads land before exit
          (void)mbar_wait(smem_u32(&s.qown_full), 0, nullptr, kDrainBudgetNs);
          (void)mbar_wait(smem_u32(&s.q_full), 0, nullptr, kDrainBudgetNs);
        }
      }
    }
  } else if (kFp8 && (warp == 10 || warp == 11)) {
    // ------------------------------------------------------------ FP8 converters
    // Warp 10 widens every tile's other part, warp 11 its own part, in tile
    // order, each from the staging half of the slot, and hands the slot to
    // the MMAs (other_full / own_full).  Before a segment's first tile, warp
    // 11 turns that segment's q own dims and rope into f16 (qown_conv), warp 10
    // its other dims (q_conv), so that every MMA operand is f16.
    if (active) {
      const bool own_part = (warp == 11);
      SegIter<kTile> it;
      it.init(v, prm.batch, pair, seg_n, seg_first);
      int32_t t0, t1, slot_p;
      uint32_t g = 0, seg = 0;
      bool ok = true;
      while (ok && it.next(t0, t1, slot_p)) {
        if (own_part) {
          if (!warp_wait(smem_u32(&s.qown_full), seg & 1u, abort_flag)) {
            if (lane == 0) set_abort(s, prm.dev_status);
            break;
          }
          for (int c = 0; c < 4; ++c)
            q_to_f16(seg == 0 ? q_stage_chunk(s, c) : s.q_other[c], kQChunkBytes, lane);
          q_to_f16(s.q_rope, kQChunkBytes, lane);
          fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&s.qown_conv));
        } else {
          if (!warp_wait(smem_u32(&s.q_full), seg & 1u, abort_flag)) {
            if (lane == 0) set_abort(s, prm.dev_status);
            break;
          }
          for (int c = 0; c < 4; ++c) q_to_f16(s.q_other[c], kQChunkBytes, lane);
          fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&s.q_conv));
        }
        ++seg;
        for (int32_t tt = t0; tt < t1; tt += kTile, ++g) {
          const int slot = g % kSlots;
          const uint32_t ph = (g / kSlots) & 1u;
          if (!warp_wait(smem_u32(own_part ? &s.own_staged[slot] : &s.other_staged[slot]), ph,
                         abort_flag)) {
            if (lane == 0) set_abort(s, prm.dev_status);
            ok = false;
            break;
          }
          // the slot as one byte array: chunks, then (upper half) the staging
          if (own_part) {
            uint8_t *slot_bytes = reinterpret_cast<uint8_t *>(s.own[slot]);
            widen_part_fp8<4>(slot_bytes, slot_bytes + kOwnStage, lane);
          } else {
            uint8_t *slot_bytes = reinterpret_cast<uint8_t *>(s.other[slot]);
            widen_part_fp8<5>(slot_bytes, slot_bytes + kOtherStage, lane);
          }
          fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(own_part ? &s.own_full[slot] : &s.other_full[slot]));
        }
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ softmax / epilogue
    const int q4 = warp & 3;              // TMEM lane quadrant of this warp
    const int h = q4 * 32 + lane;         // head = TMEM lane
    const uint32_t lane_addr = tmem + ((uint32_t)(q4 * 32) << 16);
    const int st = tid - 128;             // 0..127 within the softmax group

    // requests with no context: out = 0 (this CTA's half), lse = -inf
    for (int b = pair; b < prm.batch; b += (int)(gridDim.x >> 1)) {
      if (v.seq_len[b] != 0) continue;
      uint4 *o = (uint4 *)(prm.out + ((int64_t)b * kHeads + h) * kVDim + half * kVHalf);
#pragma unroll 4
      for (int k = 0; k < kVHalf / 8; ++k) o[k] = make_uint4(0, 0, 0, 0);
      if (prm.lse && half == 0) prm.lse[(int64_t)b * kHeads + h] = -INFINITY;
    }

    if (active && plan_ok()) {  // outputs are written where the plan's records say
      SegIter<kTile> it;
      it.init(v, prm.batch, pair, seg_n, seg_first);
      int32_t t0, t1, slot_p;
      uint32_t g = 0;  // tiles so far
      bool ok = true;
      bool have = it.next(t0, t1, slot_p);
      while (ok && have) {
        const int b = it.b;
        SegIter<kTile> nx = it;  // the segment after this one, if any
        int32_t nt0, nt1, nslot;
        const bool have_next = nx.next(nt0, nt1, nslot);

        float m_used = -INFINITY, l = 0.f;
        for (int32_t tt = t0; tt < t1; tt += kTile, ++g) {
          const int n = min(kTile, t1 - tt);
          const bool first = (tt == t0);
          const uint32_t buf_col = kColS + 64 * (g & 1u);
          if (!warp_wait(smem_u32(&s.s_full[g & 1u]), (g >> 1) & 1u, abort_flag)) {
            if (lane == 0) set_abort(s, prm.dev_status);
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t xr[kTile];
          tmem_ld32(lane_addr + buf_col, &xr[0]);
          tmem_ld32(lane_addr + buf_col + 32, &xr[32]);
          tmem_wait_ld();
          // ---- online softmax in log2 units, lazy rescale of O (eight
          // independent partial maxima / sums keep the dependency chains short).
          // The scale is positive (checked on the host), so the tile max is
          // taken on the raw scores and each exponent is one fma, s*c - m;
          // columns past the sequence end (tail tiles only) are masked.
          float x[kTile];
          float mx[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) mx[k] = -INFINITY;
          if (n == kTile) {
#pragma unroll
            for (int k = 0; k < kTile; ++k) {
              x[k] = __uint_as_float(xr[k]);
              mx[k & 7] = fmaxf(mx[k & 7], x[k]);
            }
          } else {
#pragma unroll
            for (int k = 0; k < kTile; ++k) {
              x[k] = k < n ? __uint_as_float(xr[k]) : -INFINITY;
              mx[k & 7] = fmaxf(mx[k & 7], x[k]);
            }
          }
          const float tmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                   fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) *
                             prm.scale_log2;
          const bool rescale = first || tmax > m_used + kRescaleThreshold;
          float alpha = 1.f;
          if (rescale) {
            const float m_new = first ? tmax : fmaxf(m_used, tmax);
            alpha = first ? 0.f : ex2_approx(m_used - m_new);
            m_used = m_new;
          }
          uint32_t pk[kTile / 2];
          float ps[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) ps[k] = 0.f;
          const float c = prm.scale_log2, nm = -m_used;
#pragma unroll
          for (int k = 0; k < kTile; k += 2) {
            const float p0 = ex2_approx(fmaf(x[k], c, nm)), p1 = ex2_approx(fmaf(x[k + 1], c, nm));
            ps[(k >> 1) & 7] += p0 + p1;
            pk[k / 2] = kFp8 ? pack_f16(p0, p1) : pack_bf16(p0, p1);
          }
          const float psum = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
          l = l * alpha + psum;
          // ---- O may be rescaled only once the previous P V has completed
          if (!first && __any_sync(0xffffffffu, rescale)) {
            if (!warp_wait(smem_u32(&s.pv_done[(g - 1) & 1u]), ((g - 1) >> 1) & 1u, abort_flag)) {
              if (lane == 0) set_abort(s, prm.dev_status);
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < kVHalf; c += 32) {
              uint32_t o[32];
              tmem_ld32(lane_addr + kColO + c, o);
              tmem_wait_ld();
#pragma unroll
              for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
              tmem_st32(lane_addr + kColO + c, o);
            }
          }
          // P over the first 32 columns of its own S buffer (S already read)
          tmem_st32(lane_addr + buf_col, pk);
          // The P V of a tail tile reads rows [0, ceil16(n)); rows past the
          // sequence end hold whatever the page held (maybe NaN; 0 * NaN = NaN),
          // so zero them (a 128-byte row keeps its 16-byte chunks inside itself
          // under the 128-byte swizzle).
          if (n & 15) {
            uint8_t *base = s.own[g % kSlots][0];
            const int rows = ((n + 15) & ~15) - n;
            for (int k = st; k < rows * 32; k += kSoftmaxThreads) {
              const int row = n + (k >> 5), chunk = (k >> 3) & 3, c16 = k & 7;
              *reinterpret_cast<uint4 *>(base + chunk * kChunkBytes + row * 128 + c16 * 16) =
                  make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_shared();
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(smem_u32(&s.p_full[g & 1u]));
        }
        if (!ok) break;
        // ---- epilogue: O / l of this segment, after its last P V
        const uint32_t gl = g - 1;
        if (!warp_wait(smem_u32(&s.pv_done[gl & 1u]), (gl >> 1) & 1u, abort_flag)) {
          if (lane == 0) set_abort(s, prm.dev_status);
          break;
        }
        tc_fence_after();
        // with an FP8 cache every value row carries the layer's kv_scale
        const float inv = kFp8 ? prm.kv_scale / l : 1.f / l;
        // O leaves tensor memory 32 columns a load, kEpiLoads loads per wait
        // (4 cut the 20-request step by 1%; the FP8 variant, short of
        // registers, is slower with more than one)
        constexpr int kEpiLoads = kFp8 ? 1 : 4;
        const float lse_val = (m_used + log2f(l)) * 0.69314718055994531f;
        if (slot_p < 0) {
          uint4 *dst = (uint4 *)(prm.out + ((int64_t)b * kHeads + h) * kVDim + half * kVHalf);
#pragma unroll 1
          for (int c0 = 0; c0 < kVHalf; c0 += 32 * kEpiLoads) {
            uint32_t oo[32 * kEpiLoads];
#pragma unroll
            for (int u = 0; u < kEpiLoads; ++u)
              tmem_ld32(lane_addr + kColO + c0 + 32 * u, oo + 32 * u);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < kEpiLoads; ++u) {
              const int c = c0 + 32 * u;
              const uint32_t *o = oo + 32 * u;
#pragma unroll
              for (int k = 0; k < 4; ++k)
                dst[c / 8 + k] = make_uint4(
                    pack_bf16(__uint_as_float(o[8 * k]) * inv, __uint_as_float(o[8 * k + 1]) * inv),
                    pack_bf16(__uint_as_float(o[8 * k + 2]) * inv, __uint_as_float(o[8 * k + 3]) * inv),
                    pack_bf16(__uint_as_float(o[8 * k + 4]) * inv, __uint_as_float(o[8 * k + 5]) * inv),
                    pack_bf16(__uint_as_float(o[8 * k + 6]) * inv, __uint_as_float(o[8 * k + 7]) * inv));
            }
          }
          if (prm.lse && half == 0) prm.lse[(int64_t)b * kHeads + h] = lse_val;
        } else {
          // partials are stored in bf16 as [slot][dim / 8][head][8]: a warp's
          // 32 heads of eight dims are 512 contiguous bytes, so every 16-byte
          // store coalesces (head-major rows, one per thread, cost a line per
          // lane)
          const int slot = slot_p;
          uint4 *dst = reinterpret_cast<uint4 *>(v.o_part) +
                       ((int64_t)slot * (kVDim / 8) + half * (kVHalf / 8)) * kHeads + h;
#pragma unroll 1
          for (int c0 = 0; c0 < kVHalf; c0 += 32 * kEpiLoads) {
            uint32_t oo[32 * kEpiLoads];
#pragma unroll
            for (int u = 0; u < kEpiLoads; ++u)
              tmem_ld32(lane_addr + kColO + c0 + 32 * u, oo + 32 * u);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < kEpiLoads; ++u) {
              const int c = c0 + 32 * u;
              const uint32_t *o = oo + 32 * u;
#pragma unroll
              for (int k = 0; k < 4; ++k)
                dst[(int64_t)(c / 8 + k) * kHeads] = make_uint4(
                    pack_bf16(__uint_as_float(o[8 * k]) * inv, __uint_as_float(o[8 * k + 1]) * inv),
                    pack_bf16(__uint_as_float(o[8 * k + 2]) * inv, __uint_as_float(o[8 * k + 3]) * inv),
                    pack_bf16(__uint_as_float(o[8 * k + 4]) * inv, __uint_as_float(o[8 * k + 5]) * inv),
                    pack_bf16(__uint_as_float(o[8 * k + 6]) * inv, __uint_as_float(o[8 * k + 7]) * inv));
            }
          }
          if (half == 0) v.lse_part[(int64_t)slot * kHeads + h] = lse_val;
        }
        tc_fence_before();
        // advance to the next segment (already peeked)
        it = nx;
        t0 = nt0;
        t1 = nt1;
        slot_p = nslot;
        have = have_next;
      }
    }
  }

  // ------------------------------------------------------------ teardown
  // Each warp reports the end of its role on roles_done once all its lanes
  // are here (in the role warps one elected lane worked while the others went
  // on), and the tensor memory is freed only after every report.  A CTA-wide
  // __syncthreads reached by warps in that state was measured to release some
  // warps microseconds before others had arrived, so it does not order this.
  __syncwarp();
  tc_fence_before();
  if (lane == 0) mbar_arrive(smem_u32(&s.roles_done));
  if (warp == 4) {
    // one lane polls (the others wait without taking issue slots)
    if (lane == 0 && !mbar_wait(smem_u32(&s.roles_done), 0, nullptr, kWaitBudgetNs))
      report(prm.dev_status, MLA_ERR_DEVICE_TIMEOUT);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Check of the bounded waits, without a fault or a hang: warp 0 waits on a
// barrier nothing arrives at, with budget_ns; when its wait gives up it raises
// the abort flag and reports MLA_ERR_DEVICE_TIMEOUT, as the decode's roles do.
// Warp 1 waits on another such barrier through the decode's own warp_wait
// (100 ms budget, released by the abort flag), so it returns soon after warp
// 0 gives up.  Each warp's wait time goes to elapsed_ns[warp]; the kernel
// then ends normally and the context stays usable.
__global__ void __launch_bounds__(64) wait_selftest_kernel(int32_t *dev_status, uint64_t budget_ns,
                                                           uint64_t *elapsed_ns) {
  __shared__ __align__(8) uint64_t bar[2];
  __shared__ int abort;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar[0]), 1);
    mbar_init(smem_u32(&bar[1]), 1);
    abort = 0;
    fence_mbarrier_init_cluster();
  }
  __syncthreads();
  volatile int *abort_flag = &abort;
  const uint64_t t0 = globaltimer();
  bool ok;
  if (warp == 0) {
    ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar[0]), 0, nullptr, budget_ns));
    if (!ok && lane == 0) {
      *abort_flag = 1;
      report(dev_status, MLA_ERR_DEVICE_TIMEOUT);
    }
  } else {
    ok = warp_wait(smem_u32(&bar[1]), 0, abort_flag);
  }
  if (lane == 0) elapsed_ns[warp] = ok ? 0 : globaltimer() - t0;
}

}  // namespace tc

cudaError_t launch_wait_selftest(int32_t *dev_status, uint64_t budget_ns, uint64_t *elapsed_ns,
                                 cudaStream_t stream) {
  tc::wait_selftest_kernel<<<1, 64, 0, stream>>>(dev_status, budget_ns, elapsed_ns);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------- host

int tc_unit_tokens() { return tc::kTile; }

// Split ranges of the tensor-core kernel: one per pair of SMs (two CTAs of
// one SM each work on a range).
int tc_max_pairs() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  if (cached[dev] > 0) return cached[dev];
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  cached[dev] = sms / 2 > 0 ? sms / 2 : 1;
  return cached[dev];
}

namespace {
// Tensor maps depend only on the tensor's address and shape, so they are
// encoded once and kept in small direct-mapped caches (a decode step touches
// one cache and one q tensor per layer: 61 of each for a DeepSeek-V3 step).
// Eager callers then pay no encode per call; graph replays never did.
struct KvEntry {
  bool valid;
  bool fp8;
  int dev;
  const void *base;
  int64_t rows;
  int32_t block_size;
  CUtensorMap kv5, kv4, kv1, kv2d;
};
struct QEntry {
  bool valid;
  int dev;
  const void *base;
  int32_t batch;
  CUtensorMap q;
};
constexpr int kMapCacheSize = 256;
std::mutex g_map_mu;
KvEntry g_kv_maps[kMapCacheSize];
QEntry g_q_maps[kMapCacheSize];


bool kv_maps(int dev, const void *cache, int64_t rows, int32_t block_size, bool fp8,
             tc::Maps *m) {
  std::lock_guard<std::mutex> lock(g_map_mu);
  KvEntry &e = g_kv_maps[tmap::slot_of_ptr(cache, kMapCacheSize)];
  if (!(e.valid && e.dev == dev && e.base == cache && e.rows == rows &&
        e.block_size == block_size && e.fp8 == fp8)) {
    const uint32_t box_rows = block_size < tc::kTile ? (uint32_t)block_size : (uint32_t)tc::kTile;
    e.valid = false;
    const bool ok =
        fp8 ? tmap::encode_2d_u8(&e.kv2d, cache, rows, box_rows) &&
                  tmap::encode_3d_u8(&e.kv5, cache, rows, box_rows, 5) &&
                  tmap::encode_3d_u8(&e.kv4, cache, rows, box_rows, 4) &&
                  tmap::encode_3d_u8(&e.kv1, cache, rows, box_rows, 1)
            : tmap::encode_2d(&e.kv2d, cache, rows, box_rows) &&
                  tmap::encode_3d(&e.kv5, cache, rows, box_rows, 5) &&
                  tmap::encode_3d(&e.kv4, cache, rows, box_rows, 4) &&
                  tmap::encode_3d(&e.kv1, cache, rows, box_rows, 1);
    if (!ok) return false;
    e.valid = true;
    e.fp8 = fp8;
    e.dev = dev;
    e.base = cache;
    e.rows = rows;
    e.block_size = block_size;
  }
  m->kv5 = e.kv5;
  m->kv4 = e.kv4;
  m->kv1 = e.kv1;
  m->kv2d = e.kv2d;
  return true;
}

bool q_map(int dev, const void *q, int32_t batch, tc::Maps *m) {
  std::lock_guard<std::mutex> lock(g_map_mu);
  QEntry &e = g_q_maps[tmap::slot_of_ptr(q, kMapCacheSize)];
  if (!(e.valid && e.dev == dev && e.base == q && e.batch == batch)) {
    e.valid = false;
    if (!tmap::encode_2d(&e.q, q, (int64_t)batch * kHeads, kHeads)) return false;
    e.valid = true;
    e.dev = dev;
    e.base = q;
    e.batch = batch;
  }
  m->q = e.q;
  return true;
}

// the kernel's dynamic shared memory opt-in, set once per device and cache type
template <bool kFp8>
cudaError_t ensure_smem_attr(int dev, size_t smem) {
  static std::atomic<bool> done[64];
  if (dev >= 0 && dev < 64 && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(tc::decode_tc_kernel<kFp8>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev].store(true, std::memory_order_release);
  return e;
}
}  // namespace

cudaError_t launch_decode_tc(const void *q, const void *cache, int64_t num_blocks, int32_t block_size,
                             const int32_t *block_table, int32_t max_blocks_per_seq, int32_t batch,
                             float softmax_scale, void *out, float *lse, void *ws,
                             int32_t max_ranges, int32_t *dev_status, cudaStream_t stream,
                             const void *kv_new, bool fp8, float kv_scale, bool early_launch) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  tc::Maps maps;
  if (!kv_maps(dev, cache, num_blocks * (int64_t)block_size, block_size, fp8, &maps) ||
      !q_map(dev, q, batch, &maps))
    return cudaErrorInvalidValue;
  const size_t smem = sizeof(tc::Smem) + 1024;
  e = fp8 ? ensure_smem_attr<true>(dev, smem) : ensure_smem_attr<false>(dev, smem);
  if (e != cudaSuccess) return e;
  tc::Params p;
  p.q = (const __nv_bfloat16 *)q;
  p.block_table = block_table;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.block_size = block_size;
  p.num_blocks = (int32_t)num_blocks;
  p.batch = batch;
  // with an FP8 cache the layer's kv_scale multiplies every score
  p.scale_log2 = fp8 ? softmax_scale * kv_scale * 1.4426950408889634f
                     : softmax_scale * 1.4426950408889634f;
  p.kv_scale = fp8 ? kv_scale : 1.f;
  p.kv_inv_scale = fp8 ? 1.f / kv_scale : 1.f;
  p.out = (__nv_bfloat16 *)out;
  p.lse = lse;
  p.ws = ws;
  p.max_ranges = max_ranges;
  p.dev_status = dev_status;
  p.kv_new = (const uint4 *)kv_new;
  p.cache_rows = (uint4 *)const_cast<void *>(cache);
  p.early_launch = early_launch ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * max_ranges);
  cfg.blockDim = dim3(fp8 ? tc::kThreadsFp8 : tc::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = early_launch ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return fp8 ? cudaLaunchKernelEx(&cfg, tc::decode_tc_kernel<true>, maps, p)
             : cudaLaunchKernelEx(&cfg, tc::decode_tc_kernel<false>, maps, p);
}

}  // namespace mla
