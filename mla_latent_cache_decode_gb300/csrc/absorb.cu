// The absorption GEMMs on either side of the absorbed-form decode: the query
// side maps every head's 128-dim non-rotary query into the 512-dim latent
// (q[b,h,0:512] = q_nope[b,h,:] . W_UK[h], rope dims copied behind it), the
// output side maps the latent attention output back to the head's 128 value
// dims (o[b,h,:] = out[b,h,:] . W_UV[h]).  With these, a head attends over the
// shared latent directly, which is what decode runs [dp-attention-expert-
// parallel-mla-kv-replication (inferenceinterviews.com), "A strong answer":
// "each head's query is projected into the latent space"]; qk_nope and the
// value dims are the 128 of the head, the rope dims the 64 shared ones [MLA
// 的 TP 切分 (10100.com), §2.2].
//
// Per head both are C[B x N] = A[B x K] . W[K x N] with a small batch B (a DP
// rank's requests) and a 128 KB weight: the time is the weight stream.  One
// CTA per (head, 256 or 64 columns of N, 128 rows of B) streams its weight
// slab through a TMA ring and multiplies on the tensor cores with M = 128
// (rows past B are zero-filled by TMA and never written back):
//   A  rows of B, K-major, 128-byte swizzle: boxes {64 k, 1 head, R rows},
//      R = B rounded up to 8 (at most 128); the MMA's rows past R read stale
//      shared memory, which only reaches output rows that are not written
//   W  the head's [K x N] slab, N contiguous (MN-major), 128-byte swizzle:
//      boxes {64 n, 64 k, 1 head}, N-tile / 64 of them per K chunk
//   D  fp32 in tensor memory (N-tile columns), read back by the four warps.
#include <mutex>

#include "common.cuh"
#include "sm100.cuh"
#include "trace.h"

namespace mla {
void set_error_detail(const char *msg);

namespace absorb {
using namespace sm100;

constexpr int kThreads = 128;
constexpr int kKChunk = 64;                 // K per stage
constexpr int kWBox = kKChunk * 64 * 2;     // 8 KB: 64 k rows x 64 n
constexpr int kNope = 128;                  // non-rotary query dims per head
constexpr int kRope = 64;                   // shared rotary dims
constexpr int kVHead = 128;                 // value dims per head after W_UV
constexpr uint64_t kWaitNs = 100000000ull;  // 100 ms per wait
constexpr uint64_t kDrainNs = 10000000ull;  // 10 ms to drain issued copies on abort

// Dynamic shared memory, from a 1024-byte boundary: ST stages of
// {W: NT / 64 boxes of kWBox, then A: a_rows x 128 B} (a_rows a multiple of 8,
// so every box starts on a 1024-byte boundary as the swizzle wants), then
// (128 - a_rows) x 128 B more: an M = 128 MMA reads 128 rows of A, which for
// the last stage run past its box.
__host__ __device__ constexpr int stage_bytes(int nt, int a_rows) {
  return (nt / 64) * kWBox + a_rows * 128;
}

struct Maps {
  CUtensorMap a, w;
};

struct Params {
  int32_t batch, k;            // B, K (a multiple of 64)
  int32_t a_rows;              // rows of an A box: B rounded up to 8, at most 128
  __nv_bfloat16 *c;            // C rows: c + b * ldc + h * c_head + n
  int64_t ldc, c_head;
  const __nv_bfloat16 *rope;   // absorb_q: q_pe [B][128][64], copied to c[..., 512:576]
  int32_t *dev_status;         // nullable: MLA_ERR_DEVICE_TIMEOUT when a wait runs out
};

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// grid = (N / NT, 128 heads, ceil(B / 128)), 128 threads
template <int NT, int ST>
__global__ void __launch_bounds__(kThreads) absorb_kernel(const __grid_constant__ Maps maps,
                                                          const Params prm) {
  extern __shared__ uint8_t smem_raw[];
  struct Bars {
    uint64_t full[ST], empty[ST], done;
    uint32_t tmem_base;
    int abort;  // a wait ran out: the other roles stop waiting, nothing is stored
  };
  __shared__ Bars s;
  uint8_t *stages = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int sbytes = stage_bytes(NT, prm.a_rows);
  auto w_box = [&](int st, int j) { return stages + st * sbytes + j * kWBox; };
  auto a_box = [&](int st) { return stages + st * sbytes + (NT / 64) * kWBox; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * NT, h = blockIdx.y, m0 = blockIdx.z * 128;
  const int nk = prm.k / kKChunk;
  if (threadIdx.x == 0) {
    for (int i = 0; i < ST; ++i) {
      mbar_init(smem_u32(&s.full[i]), 1);
      mbar_init(smem_u32(&s.empty[i]), 1);
    }
    mbar_init(smem_u32(&s.done), 1);
    s.abort = 0;
    fence_mbarrier_init_cluster();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(&s.tmem_base), NT);
    tmem_relinquish();
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  // Launched as a programmatic dependent: the next kernel may launch now, and
  // this one's weight loads (constant across calls) may start before the
  // previous kernel has finished.  Everything else — the activations it reads
  // and every global write — comes after griddepcontrol.wait, which returns
  // once the previous kernel has completed and its writes are visible.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // the weight slabs of the first stages, ahead of the wait
  if (warp == 0 && elect_one_sync()) {
    prefetch_tmap(&maps.w);
    for (int kc = 0; kc < nk && kc < ST; ++kc) {
      const uint32_t bar = smem_u32(&s.full[kc]);
      mbar_arrive_expect_tx(bar, (uint32_t)sbytes);
      for (int j = 0; j < NT / 64; ++j)
        tma_load_3d_hint(smem_u32(w_box(kc, j)), &maps.w, n0 + 64 * j, kc * kKChunk, h, bar,
                         policy_evict_normal());
    }
  }
  __syncwarp();
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // the rotary dims of the query, copied behind the latent ones (one CTA per
  // head and row tile: the first column tile's)
  if (prm.rope && blockIdx.x == 0) {
    const int b = m0 + threadIdx.x;
    if (b < prm.batch) {
      const uint4 *src = reinterpret_cast<const uint4 *>(prm.rope + ((int64_t)b * kHeads + h) * kRope);
      uint4 *dst = reinterpret_cast<uint4 *>(prm.c + (int64_t)b * prm.ldc + h * prm.c_head + kVDim);
#pragma unroll
      for (int i = 0; i < kRope * 2 / 16; ++i) dst[i] = __ldg(src + i);
    }
  }

  volatile int *abort_flag = &s.abort;
  auto give_up = [&]() {
    *abort_flag = 1;
    report(prm.dev_status, MLA_ERR_DEVICE_TIMEOUT);
  };
  if (warp == 0) {
    if (elect_one_sync()) {  // TMA producer
      prefetch_tmap(&maps.a);
      // stages up to min(nk, ST) had their weights requested before the wait
      int issued = 0;  // chunks whose loads are all issued
      for (int kc = 0; kc < nk; ++kc) {
        const int st = kc % ST;
        const uint32_t bar = smem_u32(&s.full[st]);
        if (kc >= ST) {  // a later stage: its slot once free, then its weights too
          if (!mbar_wait(smem_u32(&s.empty[st]), ((kc / ST) & 1u) ^ 1u, abort_flag, kWaitNs)) {
            if (!*abort_flag) give_up();
            break;
          }
          mbar_arrive_expect_tx(bar, (uint32_t)sbytes);
          for (int j = 0; j < NT / 64; ++j)
            tma_load_3d_hint(smem_u32(w_box(st, j)), &maps.w, n0 + 64 * j, kc * kKChunk, h, bar,
                             policy_evict_normal());
        }
        tma_load_3d_hint(smem_u32(a_box(st)), &maps.a, kc * kKChunk, h, m0, bar,
                         policy_evict_normal());
        issued = kc + 1;
      }
      if (*abort_flag) {
        // no copy may still be landing when the shared memory is given up:
        // wait (bounded) for the last chunk issued into each stage
        for (int st = 0; st < ST && st < issued; ++st) {
          const int last = st + ((issued - 1 - st) / ST) * ST;
          (void)mbar_wait(smem_u32(&s.full[st]), (last / ST) & 1u, nullptr, kDrainNs);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (elect_one_sync()) {  // MMA issuer
      const uint32_t id = idesc_bf16_f32(128, NT, 1);
      for (int kc = 0; kc < nk; ++kc) {
        const int st = kc % ST;
        if (!mbar_wait(smem_u32(&s.full[st]), (kc / ST) & 1u, abort_flag, kWaitNs)) {
          if (!*abort_flag) give_up();
          break;
        }
        tc_fence_after();
        const uint64_t da = smem_desc(smem_u32(a_box(st)), 16, 1024, kSwizzle128B);
        const uint64_t dw = smem_desc(smem_u32(w_box(st, 0)), kWBox, 1024, kSwizzle128B);
#pragma unroll
        for (int kk = 0; kk < kKChunk / 16; ++kk)
          mma_ss(tmem, da + (uint64_t)((kk * 32) >> 4), dw + (uint64_t)((kk * 2048) >> 4), id,
                 (kc > 0 || kk > 0) ? 1u : 0u);
        mma_commit(smem_u32(&s.empty[st]));
      }
      // also after an abort: done then marks the completion of every MMA
      // issued, so the tensor memory is freed only once they are finished
      mma_commit(smem_u32(&s.done));
    }
    __syncwarp();
  }

  // epilogue: warp w holds rows m0 + 32w .. m0 + 32w + 31 in its TMEM lanes
  const bool done = mbar_wait(smem_u32(&s.done), 0, nullptr, kWaitNs);
  if (!done && lane == 0) report(prm.dev_status, MLA_ERR_DEVICE_TIMEOUT);
  if (__all_sync(0xffffffffu, done) && !*abort_flag && m0 + 32 * warp < prm.batch) {
    tc_fence_after();
    const int b = m0 + 32 * warp + lane;
    __nv_bfloat16 *row = prm.c + (int64_t)b * prm.ldc + h * prm.c_head + n0;
#pragma unroll 1
    for (int c = 0; c < NT; c += 32) {
      uint32_t r[32];
      tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + c, r);
      tmem_wait_ld();
      if (b < prm.batch) {
        uint4 *dst = reinterpret_cast<uint4 *>(row + c);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          dst[i] = make_uint4(pack2(__uint_as_float(r[8 * i]), __uint_as_float(r[8 * i + 1])),
                              pack2(__uint_as_float(r[8 * i + 2]), __uint_as_float(r[8 * i + 3])),
                              pack2(__uint_as_float(r[8 * i + 4]), __uint_as_float(r[8 * i + 5])),
                              pack2(__uint_as_float(r[8 * i + 6]), __uint_as_float(r[8 * i + 7])));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, NT);
  }
}

}  // namespace absorb

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)p;
  });
  return fn;
}

// A bf16 3-D tensor {d0 (contiguous), d1, d2} with byte strides s1, s2, read
// in boxes {b0, b1, b2} with the 128-byte swizzle (b0 * 2 = 128 B); elements
// outside the tensor read as zero.
bool encode(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
            uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1, s2};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// Encoded maps kept in a small direct-mapped cache keyed by the tensor's
// address and shape (a step touches two weights per layer and the same few
// activations), so that eager callers do not encode at every call.
struct MapEntry {
  bool valid;
  int dev;
  const void *base;
  uint64_t d0, d1, d2;
  uint32_t b2;
  CUtensorMap map;
};
MapEntry g_maps[512];
std::mutex g_maps_mu;

bool cached_encode(CUtensorMap *m, int dev, const void *base, uint64_t d0, uint64_t d1,
                   uint64_t d2, uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2) {
  std::lock_guard<std::mutex> lock(g_maps_mu);
  MapEntry &e = g_maps[(((uintptr_t)base >> 8) ^ (d0 * 31 + d2)) % 512];
  if (!(e.valid && e.dev == dev && e.base == base && e.d0 == d0 && e.d1 == d1 && e.d2 == d2 &&
        e.b2 == b2)) {
    e.valid = false;
    if (!encode(&e.map, base, d0, d1, d2, s1, s2, b0, b1, b2)) return false;
    e.valid = true;
    e.dev = dev;
    e.base = base;
    e.d0 = d0;
    e.d1 = d1;
    e.d2 = d2;
    e.b2 = b2;
  }
  *m = e.map;
  return true;
}

template <int NT, int ST>
cudaError_t launch(const void *a, int k, const void *w, int n, int batch, void *c, int64_t ldc,
                   int64_t c_head, const void *rope, int32_t *dev_status, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  absorb::Maps maps;
  // A [B][128 heads][K]: boxes {64 k, 1 head, a_rows rows}
  // W [128 heads][K][N]: boxes {64 n, 64 k, 1 head}
  const int a_rows = batch >= 128 ? 128 : (batch + 7) / 8 * 8;
  if (!cached_encode(&maps.a, dev, a, k, kHeads, batch, (uint64_t)k * 2,
                     (uint64_t)kHeads * k * 2, 64, 1, a_rows) ||
      !cached_encode(&maps.w, dev, w, n, k, kHeads, (uint64_t)n * 2, (uint64_t)k * n * 2, 64, 64,
                     1))
    return cudaErrorInvalidValue;
  const size_t smem = (size_t)ST * absorb::stage_bytes(NT, a_rows) + (128 - a_rows) * 128 + 1024;
  const size_t smem_max = (size_t)ST * absorb::stage_bytes(NT, 128) + 1024;
  static std::once_flag attr_once[64];
  std::call_once(attr_once[dev], [&] {
    e = cudaFuncSetAttribute(absorb::absorb_kernel<NT, ST>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_max);
  });
  if (e != cudaSuccess) return e;
  absorb::Params p;
  p.batch = batch;
  p.k = k;
  p.a_rows = a_rows;
  p.c = (__nv_bfloat16 *)c;
  p.ldc = ldc;
  p.c_head = c_head;
  p.rope = (const __nv_bfloat16 *)rope;
  p.dev_status = dev_status;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n / NT, kHeads, (batch + 127) / 128);
  cfg.blockDim = dim3(absorb::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, absorb::absorb_kernel<NT, ST>, maps, p);
}

mla_status_t check(const void *const *ptrs, int count, int32_t batch, int32_t num_heads) {
  if (batch < 0) {
    set_error_detail("batch < 0");
    return MLA_ERR_INVALID_ARGUMENT;
  }
  if (num_heads != kHeads) {
    set_error_detail("num_heads must be 128");
    return MLA_ERR_UNSUPPORTED;
  }
  if (batch == 0) return MLA_OK;
  for (int i = 0; i < count; ++i) {
    if (!ptrs[i]) {
      set_error_detail("null pointer");
      return MLA_ERR_INVALID_ARGUMENT;
    }
    if (!aligned16(ptrs[i])) {
      set_error_detail("pointers must be 16-byte aligned");
      return MLA_ERR_INVALID_ARGUMENT;
    }
  }
  return MLA_OK;
}

mla_status_t launched(cudaError_t e) {
  if (e == cudaSuccess) return MLA_OK;
  set_error_detail(cudaGetErrorString(e));
  return MLA_ERR_CUDA;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" {

mla_status_t mla_absorb_q(const void *q_nope, const void *q_pe, const void *w_uk, int32_t batch,
                          int32_t num_heads, void *q, int32_t *dev_status, void *stream) {
  TraceRange trace_range("mla_absorb_q");
  set_error_detail("");
  const void *ptrs[4] = {q_nope, q_pe, w_uk, q};
  mla_status_t s = check(ptrs, 4, batch, num_heads);
  if (s != MLA_OK || batch == 0) return s;
  // q[b, h, 0:512] = q_nope[b, h, :] . W_UK[h]; q[b, h, 512:576] = q_pe[b, h, :]
  // 256 columns a CTA, the whole K (two chunks) in flight
  return launched(launch<256, 2>(q_nope, absorb::kNope, w_uk, kVDim, batch, q, (int64_t)kHeads * kRow,
                              kRow, q_pe, dev_status, (cudaStream_t)stream));
}

mla_status_t mla_absorb_out(const void *out, const void *w_uv, int32_t batch, int32_t num_heads,
                            void *o, int32_t *dev_status, void *stream) {
  TraceRange trace_range("mla_absorb_out");
  set_error_detail("");
  const void *ptrs[3] = {out, w_uv, o};
  mla_status_t s = check(ptrs, 3, batch, num_heads);
  if (s != MLA_OK || batch == 0) return s;
  // o[b, h, :] = out[b, h, :] . W_UV[h]
  // 64 columns a CTA (two per head), the whole K (eight chunks) in flight
  return launched(launch<64, 8>(out, kVDim, w_uv, absorb::kVHead, batch, o,
                              (int64_t)kHeads * absorb::kVHead, absorb::kVHead, nullptr,
                              dev_status, (cudaStream_t)stream));
}

}  // extern "C"
