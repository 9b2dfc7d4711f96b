// Tensor-core MLA decode for sm_103a (tcgen05 + TMA + mbarrier pipeline).
//
// What is computed: absorbed-form MLA decode over the shared latent.  Every
// head's score uses all 576 dims of each cached row (512 kv_c + 64 k_rope
// shared by all heads) and the output is the softmax-weighted sum of the
// 512-dim kv_c  [dp-attention-expert-parallel-mla-kv-replication
// (inferenceinterviews.com), "A strong answer"; MLA 的 TP 切分 (10100.com),
// sections 2.2 and 3.1; DP 与 DPA 的区别 (chengxuchu.com), v_head_dim =
// kv_lora_rank].  Because all 128 heads read the same row, the step is a dense
// contraction: S = Q K^T is [128 x 576] x [576 x tokens] and O = P V is
// [128 x tokens] x [tokens x 512], run on the tensor cores.
//
// How (one CTA pair = one cluster per split range of the plan):
//   - The pair splits the OUTPUT dims: CTA r owns O[:, 256r .. 256r+255] in
//     tensor memory (256 fp32 columns) and loads only the columns it needs of
//     every cache row: kv_c [256r, 256r+256) and rope [512+32r, 512+32r+32),
//     288 of the 576 dims.  No byte of the cache is loaded twice.
//   - Each CTA computes the partial score over its 288 dims, S_r = Q_r K_r^T
//     (M = 128 heads, N = 64 tokens, K = 288), sends it to the peer with
//     st.async into the peer's shared memory, and adds the peer's partial:
//     both CTAs then hold the same full S (fp32 addition commutes) and take
//     identical softmax decisions.
//   - Q_r (128 x 288 bf16) and P (128 x 64 bf16) live in tensor memory as the
//     A operand, so the tensor core reads only the cache tile from shared
//     memory (64 B/clk at full rate).
//   - Warp roles: warp 0 issues TMA loads of paged tiles through a 4-stage
//     mbarrier ring; warp 1 issues the MMAs; warps 2-5 (one thread per head)
//     run the exchange, an online softmax with lazy rescaling of O, and the
//     epilogue.
//   - Split-KV: a request spanning several plan ranges leaves fp32 partials
//     (normalised O and its log-sum-exp), merged by the combine kernel.
#include "common.cuh"
#include "sm100.cuh"

namespace mla {
namespace tc {

using namespace sm100;

constexpr int kTile = 64;                 // tokens per tile (= plan unit)
constexpr int kStages = 4;
constexpr int kVHalf = 256;               // output dims per CTA
constexpr int kRopeHalf = 32;             // rope dims per CTA
constexpr int kRegionBytes = kTile * 128; // one 64-dim SW128 region of a tile: 8 KB
constexpr int kRopeBytes = kTile * 64;    // the 32-dim SW64 rope region: 4 KB
constexpr int kStageBytes = 4 * kRegionBytes + kRopeBytes;  // 36 KB
constexpr int kRecvStride = kTile + 4;    // floats per received row (16 B pad)
constexpr int kThreads = 192;             // 6 warps
constexpr int kSoftmaxThreads = 128;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 256, kColP = 320, kColQ = 352;
constexpr uint64_t kWaitBudgetNs = 100000000ull;  // 100 ms per wait, far above any legal wait
constexpr uint64_t kDrainBudgetNs = 10000000ull;  // 10 ms to drain in-flight copies on abort
constexpr float kRescaleThreshold = 8.0f;         // log2 units

struct __align__(1024) Smem {
  uint8_t stage[kStages][kStageBytes];
  float recv[2][kSoftmaxThreads][kRecvStride];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t s_full, s_free, p_full, pv_done, q_ready, fin;
  uint64_t recv_full[2];
  uint64_t send_ok[2];
  uint32_t tmem_base;
  int abort;
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
};

// Segment of range p: request b, tokens [t0, t1).  Iterates in plan order.
struct SegIter {
  PlanView v;
  int32_t batch, U, P, r0, r1, b;
  __device__ void init(const PlanView &pv, int32_t batch_, int32_t p) {
    v = pv;
    batch = batch_;
    U = v.hdr->total_units;
    P = v.hdr->num_ranges;
    r0 = range_begin(p, U, P);
    r1 = range_begin(p + 1, U, P);
    b = v.range_first[p] - 1;
  }
  __device__ bool next(int32_t &t0, int32_t &t1, bool &split, int32_t &Ub) {
    for (++b; b < batch; ++b) {
      Ub = v.unit_prefix[b];
      if (Ub >= r1) return false;
      const int32_t Ue = v.unit_prefix[b + 1];
      const int32_t u0 = max(r0, Ub), u1 = min(r1, Ue);
      if (u0 >= u1) continue;
      t0 = (u0 - Ub) * kTile;
      t1 = min((u1 - Ub) * kTile, v.seq_len[b]);
      split = range_of(Ub, U, P) != range_of(Ue - 1, U, P);
      return true;
    }
    return false;
  }
};

__device__ __forceinline__ void set_abort(Smem &s, int32_t *dev_status) {
  s.abort = 1;
  report(dev_status, MLA_ERR_DEVICE_TIMEOUT);
}

// Every lane polls (each gets the barrier's acquire), then the warp agrees:
// the warp proceeds only if every lane saw the phase complete, so control flow
// around warp-collective tcgen05 instructions stays uniform.
template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const volatile int *abort) {
  const bool ok = mbar_wait<kCluster>(bar, parity, abort, kWaitBudgetNs);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap map_v,
                     const __grid_constant__ CUtensorMap map_r, const Params prm) {
  extern __shared__ uint8_t smem_raw[];
  Smem &s = *reinterpret_cast<Smem *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
  const int pair = blockIdx.x >> 1;
  const PlanView v = plan_view(prm.ws, prm.batch, kHeads, prm.max_ranges);
  const volatile int *abort_flag = &s.abort;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&s.full[i]), 1);
      mbar_init(smem_u32(&s.empty[i]), 1);
    }
    mbar_init(smem_u32(&s.s_full), 1);
    mbar_init(smem_u32(&s.s_free), kSoftmaxThreads);
    mbar_init(smem_u32(&s.p_full), kSoftmaxThreads);
    mbar_init(smem_u32(&s.pv_done), 1);
    mbar_init(smem_u32(&s.q_ready), kSoftmaxThreads);
    mbar_init(smem_u32(&s.fin), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s.recv_full[i]), 1);
      mbar_init(smem_u32(&s.send_ok[i]), kSoftmaxThreads / 32);  // one arrival per peer warp
    }
    s.abort = 0;
    fence_mbarrier_init_cluster();
    prefetch_tmap(&map_v);
    prefetch_tmap(&map_r);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&s.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barriers of both CTAs initialised before any remote access
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;

  const int32_t P = v.hdr->num_ranges;
  const bool active = pair < P;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (active && elect_one_sync()) {
      const uint64_t policy = policy_evict_first();
      SegIter it;
      it.init(v, prm.batch, pair);
      int32_t t0, t1, Ub;
      bool split;
      int stage = 0;
      uint32_t phase = 0;
      const int BS = prm.block_size;
      const int box_rows = BS < kTile ? BS : kTile;
      const int64_t nb = prm.num_blocks;
      bool ok = true;
      uint32_t issued = 0;
      while (ok && it.next(t0, t1, split, Ub)) {
        const int32_t *table = prm.block_table + (int64_t)it.b * prm.max_blocks_per_seq;
        for (int32_t tt = t0; tt < t1 && ok; tt += kTile) {
          const int n = min(kTile, t1 - tt);
          if (!mbar_wait(smem_u32(&s.empty[stage]), phase ^ 1u, abort_flag, kWaitBudgetNs)) {
            set_abort(s, prm.dev_status);
            ok = false;
            break;
          }
          const int boxes = (n + box_rows - 1) / box_rows;
          const uint32_t full = smem_u32(&s.full[stage]);
          mbar_arrive_expect_tx(full, (uint32_t)(boxes * box_rows * (4 * 128 + 64)));
          const uint32_t base = smem_u32(s.stage[stage]);
          for (int j = 0; j < boxes; ++j) {
            const int32_t tok = tt + j * box_rows;
            int32_t blk = table[tok / BS];
            if (blk < 0 || blk >= nb) {
              report(prm.dev_status, MLA_ERR_DEVICE_RANGE);
              blk = 0;
            }
            const int32_t y = blk * BS + (tok % BS);
            for (int c = 0; c < 4; ++c)
              tma_load_2d_hint(base + c * kRegionBytes + j * box_rows * 128, &map_v,
                               (int)rank * kVHalf + 64 * c, y, full, policy);
            tma_load_2d_hint(base + 4 * kRegionBytes + j * box_rows * 64, &map_r,
                             512 + (int)rank * kRopeHalf, y, full, policy);
          }
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (s.abort) {
        // the consumer gave up: let the last (up to kStages) issued loads land
        // before this CTA's shared memory can be released
        for (uint32_t k = 1; k <= (issued < kStages ? issued : (uint32_t)kStages); ++k) {
          const uint32_t g = issued - k;
          (void)mbar_wait(smem_u32(&s.full[g % kStages]), (g / kStages) & 1u, nullptr,
                          kDrainBudgetNs);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (active && elect_one_sync()) {
      SegIter it;
      it.init(v, prm.batch, pair);
      int32_t t0, t1, Ub;
      bool split;
      int stage = 0;
      uint32_t phase = 0;
      uint32_t q_ph = 0, s_free_ph = 0, p_full_ph = 0;
      uint32_t qk_issued = 0;
      const uint32_t id_qk = idesc_bf16_f32(128, kTile, 0);
      const uint32_t id_pv = idesc_bf16_f32(128, kVHalf, 1);
      bool ok = true;
      while (ok && it.next(t0, t1, split, Ub)) {
        if (!mbar_wait(smem_u32(&s.q_ready), q_ph, abort_flag, kWaitBudgetNs)) {
          set_abort(s, prm.dev_status);
          break;
        }
        q_ph ^= 1u;
        tc_fence_after();
        const int ntiles = (t1 - t0 + kTile - 1) / kTile;
        int prev_stage = 0, prev_n = 0;
        for (int i = 0; i <= ntiles && ok; ++i) {
          if (i < ntiles) {
            // ---- S = Q_r K_r^T for tile i
            if (!mbar_wait(smem_u32(&s.full[stage]), phase, abort_flag, kWaitBudgetNs)) {
              set_abort(s, prm.dev_status);
              ok = false;
              break;
            }
            if (qk_issued > 0) {
              if (!mbar_wait(smem_u32(&s.s_free), s_free_ph, abort_flag, kWaitBudgetNs)) {
                set_abort(s, prm.dev_status);
                ok = false;
                break;
              }
              s_free_ph ^= 1u;
            }
            tc_fence_after();
            const uint32_t base = smem_u32(s.stage[stage]);
            for (int c = 0; c < 4; ++c)
              for (int kk = 0; kk < 4; ++kk)
                mma_ts(tmem + kColS, tmem + kColQ + c * 32 + kk * 8,
                       smem_desc(base + c * kRegionBytes + kk * 32, 16, 1024, kSwizzle128B), id_qk,
                       (c | kk) != 0);
            for (int kk = 0; kk < 2; ++kk)
              mma_ts(tmem + kColS, tmem + kColQ + 128 + kk * 8,
                     smem_desc(base + 4 * kRegionBytes + kk * 32, 16, 512, kSwizzle64B), id_qk, 1);
            mma_commit(smem_u32(&s.s_full));
            ++qk_issued;
          }
          if (i > 0) {
            // ---- O += P V for tile i-1
            if (!mbar_wait(smem_u32(&s.p_full), p_full_ph, abort_flag, kWaitBudgetNs)) {
              set_abort(s, prm.dev_status);
              ok = false;
              break;
            }
            p_full_ph ^= 1u;
            tc_fence_after();
            const uint32_t base = smem_u32(s.stage[prev_stage]);
            const int ksteps = (prev_n + 15) / 16;
            for (int kt = 0; kt < ksteps; ++kt)
              mma_ts(tmem + kColO, tmem + kColP + kt * 8,
                     smem_desc(base + kt * 2048, kRegionBytes, 1024, kSwizzle128B), id_pv,
                     (i > 1 || kt > 0) ? 1u : 0u);
            mma_commit(smem_u32(&s.pv_done));
            mma_commit(smem_u32(&s.empty[prev_stage]));
          }
          if (i < ntiles) {
            prev_stage = stage;
            prev_n = min(kTile, t1 - (t0 + i * kTile));
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // all issued MMAs complete before teardown (not cut short by the abort flag)
      mma_commit(smem_u32(&s.fin));
      if (!mbar_wait(smem_u32(&s.fin), 0, nullptr, kWaitBudgetNs)) report(prm.dev_status, MLA_ERR_DEVICE_TIMEOUT);
    }
  } else {
    // ------------------------------------------------------------ softmax / exchange / epilogue
    const int q4 = warp & 3;                  // TMEM lane quadrant of this warp
    const int h = q4 * 32 + lane;             // head = TMEM lane
    const uint32_t lane_addr = tmem + ((uint32_t)(q4 * 32) << 16);
    const int st = tid - 64;                  // 0..127 within the softmax group

    // requests with no context: out = 0 (this CTA's half), lse = -inf
    for (int b = pair; b < prm.batch; b += (int)(gridDim.x >> 1)) {
      if (v.seq_len[b] != 0) continue;
      uint4 *o = (uint4 *)(prm.out + ((int64_t)b * kHeads + h) * kVDim + rank * kVHalf);
#pragma unroll 4
      for (int k = 0; k < kVHalf / 8; ++k) o[k] = make_uint4(0, 0, 0, 0);
      if (prm.lse && rank == 0) prm.lse[(int64_t)b * kHeads + h] = -INFINITY;
    }

    if (active) {
      SegIter it;
      it.init(v, prm.batch, pair);
      int32_t t0, t1, Ub;
      bool split;
      uint32_t s_full_ph = 0, pv_ph = 0;
      uint32_t xcount = 0;   // score exchanges so far (alternating buffers)
      uint32_t gtile = 0;    // tiles so far (the smem stage of a tile is gtile % kStages)
      const uint32_t my_recv[2] = {smem_u32(&s.recv[0][st][0]), smem_u32(&s.recv[1][st][0])};
      const uint32_t peer_recv[2] = {mapa_shared(my_recv[0], peer), mapa_shared(my_recv[1], peer)};
      const uint32_t peer_recv_full[2] = {mapa_shared(smem_u32(&s.recv_full[0]), peer),
                                          mapa_shared(smem_u32(&s.recv_full[1]), peer)};
      const uint32_t peer_send_ok[2] = {mapa_shared(smem_u32(&s.send_ok[0]), peer),
                                        mapa_shared(smem_u32(&s.send_ok[1]), peer)};
      bool ok = true;
      while (ok && it.next(t0, t1, split, Ub)) {
        const int b = it.b;
        // ---- Q_r of request b into tensor memory (A operand): 144 columns
        {
          const uint4 *qrow = (const uint4 *)(prm.q + ((int64_t)b * kHeads + h) * kRow);
          uint4 buf[36];
#pragma unroll
          for (int k = 0; k < 32; ++k) buf[k] = __ldg(qrow + rank * 32 + k);        // kv_c half
#pragma unroll
          for (int k = 0; k < 4; ++k) buf[32 + k] = __ldg(qrow + 64 + rank * 4 + k);  // rope half
#pragma unroll
          for (int c = 0; c < 9; ++c)
            tmem_st16(lane_addr + kColQ + 16 * c, reinterpret_cast<const uint32_t *>(&buf[4 * c]));
          tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&s.q_ready));

        float m_used = -INFINITY, l = 0.f;
        const int ntiles = (t1 - t0 + kTile - 1) / kTile;
        for (int i = 0; i < ntiles; ++i, ++gtile) {
          const int n = min(kTile, t1 - (t0 + i * kTile));
          // ---- own partial scores S_r (fp32) out of tensor memory
          if (!warp_wait(smem_u32(&s.s_full), s_full_ph, abort_flag)) {
            if (lane == 0) set_abort(s, prm.dev_status);
            ok = false;
            break;
          }
          s_full_ph ^= 1u;
          tc_fence_after();
          uint32_t xr[kTile];
          tmem_ld32(lane_addr + kColS, &xr[0]);
          tmem_ld32(lane_addr + kColS + 32, &xr[32]);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(smem_u32(&s.s_free));
          // ---- send S_r to the peer, receive S_peer
          const int xb = xcount & 1;
          const uint32_t use = xcount >> 1;
          if (use > 0 && !warp_wait<true>(smem_u32(&s.send_ok[xb]), (use - 1) & 1u, abort_flag)) {
            if (lane == 0) set_abort(s, prm.dev_status);
            ok = false;
            break;
          }
#pragma unroll
          for (int k = 0; k < kTile; k += 4)
            st_async_v4(peer_recv[xb] + 4 * k, xr[k], xr[k + 1], xr[k + 2], xr[k + 3],
                        peer_recv_full[xb]);
          if (st == 0)
            mbar_arrive_expect_tx(smem_u32(&s.recv_full[xb]),
                                  kSoftmaxThreads * kTile * (uint32_t)sizeof(float));
          if (!warp_wait<true>(smem_u32(&s.recv_full[xb]), use & 1u, abort_flag)) {
            if (lane == 0) set_abort(s, prm.dev_status);
            ok = false;
            break;
          }
          float x[kTile];
          {
            const float4 *pr = reinterpret_cast<const float4 *>(&s.recv[xb][st][0]);
#pragma unroll
            for (int k = 0; k < kTile / 4; ++k) {
              const float4 y = pr[k];
              x[4 * k] = __uint_as_float(xr[4 * k]) + y.x;
              x[4 * k + 1] = __uint_as_float(xr[4 * k + 1]) + y.y;
              x[4 * k + 2] = __uint_as_float(xr[4 * k + 2]) + y.z;
              x[4 * k + 3] = __uint_as_float(xr[4 * k + 3]) + y.w;
            }
          }
          // this warp's rows of recv[xb] are consumed: the peer may refill them
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(peer_send_ok[xb]);
          ++xcount;
          // ---- online softmax in log2 units, lazy rescale of O
          float tmax = -INFINITY;
#pragma unroll
          for (int k = 0; k < kTile; ++k) {
            x[k] = k < n ? x[k] * prm.scale_log2 : -INFINITY;
            tmax = fmaxf(tmax, x[k]);
          }
          const bool first = (i == 0);
          const bool rescale = first || tmax > m_used + kRescaleThreshold;
          float alpha = 1.f;
          if (rescale) {
            const float m_new = first ? tmax : fmaxf(m_used, tmax);
            alpha = first ? 0.f : exp2f(m_used - m_new);
            m_used = m_new;
          }
          uint32_t pk[kTile / 2];
          float psum = 0.f;
#pragma unroll
          for (int k = 0; k < kTile; k += 2) {
            const float p0 = exp2f(x[k] - m_used), p1 = exp2f(x[k + 1] - m_used);
            psum += p0 + p1;
            pk[k / 2] = pack_bf16(p0, p1);
          }
          l = l * alpha + psum;
          // ---- P and O may be touched only after the previous PV completed
          if (!first) {
            if (!warp_wait(smem_u32(&s.pv_done), pv_ph, abort_flag)) {
              if (lane == 0) set_abort(s, prm.dev_status);
              ok = false;
              break;
            }
            pv_ph ^= 1u;
            tc_fence_after();
            if (__any_sync(0xffffffffu, rescale)) {
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
          }
          tmem_st32(lane_addr + kColP, pk);
          // the PV of a tail tile reads rows [0, ceil16(n)): rows past the
          // sequence end hold whatever the page held (maybe NaN; 0 * NaN = NaN),
          // so zero them in shared memory (a 128-byte row keeps its 16-byte
          // chunks inside itself under the 128-byte swizzle)
          if (n & 15) {
            uint8_t *base = s.stage[gtile % kStages];
            const int rows = ((n + 15) & ~15) - n;
            for (int k = st; k < rows * 32; k += kSoftmaxThreads) {
              const int row = n + (k >> 5), region = (k >> 3) & 3, c16 = k & 7;
              *reinterpret_cast<uint4 *>(base + region * kRegionBytes + row * 128 + c16 * 16) =
                  make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_shared();
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(smem_u32(&s.p_full));
        }
        if (!ok) break;
        // ---- epilogue: O / l of this segment
        if (!warp_wait(smem_u32(&s.pv_done), pv_ph, abort_flag)) {
          if (lane == 0) set_abort(s, prm.dev_status);
          break;
        }
        pv_ph ^= 1u;
        tc_fence_after();
        const float inv = 1.f / l;
        const float lse_val = (m_used + log2f(l)) * 0.69314718055994531f;
        if (!split) {
          uint4 *dst = (uint4 *)(prm.out + ((int64_t)b * kHeads + h) * kVDim + rank * kVHalf);
#pragma unroll 1
          for (int c = 0; c < kVHalf; c += 32) {
            uint32_t o[32];
            tmem_ld32(lane_addr + kColO + c, o);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 4; ++k)
              dst[c / 8 + k] = make_uint4(
                  pack_bf16(__uint_as_float(o[8 * k]) * inv, __uint_as_float(o[8 * k + 1]) * inv),
                  pack_bf16(__uint_as_float(o[8 * k + 2]) * inv, __uint_as_float(o[8 * k + 3]) * inv),
                  pack_bf16(__uint_as_float(o[8 * k + 4]) * inv, __uint_as_float(o[8 * k + 5]) * inv),
                  pack_bf16(__uint_as_float(o[8 * k + 6]) * inv, __uint_as_float(o[8 * k + 7]) * inv));
          }
          if (prm.lse && rank == 0) prm.lse[(int64_t)b * kHeads + h] = lse_val;
        } else {
          const int slot = partial_slot(pair, it.U, it.P, Ub);
          float4 *dst = (float4 *)(v.o_part + ((int64_t)slot * kHeads + h) * kVDim + rank * kVHalf);
#pragma unroll 1
          for (int c = 0; c < kVHalf; c += 32) {
            uint32_t o[32];
            tmem_ld32(lane_addr + kColO + c, o);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 8; ++k)
              dst[c / 4 + k] = make_float4(
                  __uint_as_float(o[4 * k]) * inv, __uint_as_float(o[4 * k + 1]) * inv,
                  __uint_as_float(o[4 * k + 2]) * inv, __uint_as_float(o[4 * k + 3]) * inv);
          }
          if (rank == 0) v.lse_part[(int64_t)slot * kHeads + h] = lse_val;
        }
        tc_fence_before();
      }
      if (!ok || s.abort) {
        // on abort, wait (briefly) for any score the peer is still sending us
        (void)mbar_wait<true>(smem_u32(&s.recv_full[xcount & 1]), (xcount >> 1) & 1u, nullptr,
                              kDrainBudgetNs);
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no DSMEM traffic from the peer may outlive this CTA
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace tc

// ---------------------------------------------------------------------------- host

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)p;
  }
  return fn;
}

bool encode_cache_map(CUtensorMap *m, const void *cache, int64_t rows, uint32_t box_cols,
                      uint32_t box_rows, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kRow, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kRow * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(cache), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

int tc_unit_tokens() { return tc::kTile; }

// CTA pairs of the tensor-core kernel that can be resident at once on the
// current device (clusters of 2 need both SMs in one GPC), capped at SMs / 2.
int tc_max_pairs() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  if (cached[dev] > 0) return cached[dev];
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  const size_t smem = sizeof(tc::Smem) + 1024;
  if (cudaFuncSetAttribute(tc::decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return -1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
  cfg.blockDim = dim3(tc::kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, tc::decode_tc_kernel, &cfg) != cudaSuccess ||
      clusters <= 0)
    clusters = sms / 2;
  cached[dev] = clusters < sms / 2 ? clusters : sms / 2;
  return cached[dev];
}

size_t tc_smem_bytes() { return sizeof(tc::Smem) + 1024; }

cudaError_t launch_decode_tc(const void *q, const void *cache, int64_t num_blocks, int32_t block_size,
                             const int32_t *block_table, int32_t max_blocks_per_seq, int32_t batch,
                             float softmax_scale, void *out, float *lse, void *ws,
                             int32_t max_ranges, int32_t *dev_status, cudaStream_t stream) {
  CUtensorMap map_v, map_r;
  const uint32_t box_rows = block_size < tc::kTile ? (uint32_t)block_size : (uint32_t)tc::kTile;
  const int64_t rows = num_blocks * (int64_t)block_size;
  if (!encode_cache_map(&map_v, cache, rows, 64, box_rows, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_cache_map(&map_r, cache, rows, 32, box_rows, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  const size_t smem = tc_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(tc::decode_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  tc::Params p;
  p.q = (const __nv_bfloat16 *)q;
  p.block_table = block_table;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.block_size = block_size;
  p.num_blocks = (int32_t)num_blocks;
  p.batch = batch;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.out = (__nv_bfloat16 *)out;
  p.lse = lse;
  p.ws = ws;
  p.max_ranges = max_ranges;
  p.dev_status = dev_status;
  tc::decode_tc_kernel<<<2 * max_ranges, tc::kThreads, smem, stream>>>(map_v, map_r, p);
  return cudaGetLastError();
}

}  // namespace mla
