// mla_decode_noalloc: the decode entry point for callers that cannot allocate
// device memory.  Its scratch (split plan + partial results) lives in a fixed,
// file-scope device array instead of a caller-provided workspace.
#include <cuda.h>

#include <cmath>
#include <mutex>

#include "common.cuh"

namespace mla {
cudaError_t launch_plan(const int32_t *seq_lens, const int32_t *block_table, int64_t num_blocks,
                        int32_t batch, int32_t unit_tokens, int32_t max_blocks_per_seq,
                        int32_t block_size, int32_t max_ranges, void *ws, int32_t heads,
                        int32_t *dev_status, cudaStream_t stream);
cudaError_t launch_plan_combine(void *ws, int32_t batch, int32_t heads, int32_t max_ranges,
                                void *out, float *lse, cudaStream_t stream, bool early);
int tc_unit_tokens();
int tc_max_pairs();
cudaError_t launch_decode_tc(const void *q, const void *cache, int64_t num_blocks, int32_t block_size,
                             const int32_t *block_table, int32_t max_blocks_per_seq, int32_t batch,
                             float softmax_scale, void *out, float *lse, void *ws,
                             int32_t max_ranges, int32_t *dev_status, cudaStream_t stream,
                             const void *kv_new = nullptr, bool fp8 = false, float kv_scale = 1.f,
                             bool early_launch = false);
mla_status_t noalloc_fail(mla_status_t s, const char *msg);
}  // namespace mla

// Every GPU that loads this library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MLA_NOALLOC_SCRATCH_BYTES];

namespace {

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

// Unique id of the current CUDA context (0 if it cannot be read).  A context
// that is destroyed and created again (cudaDeviceReset, then any runtime call)
// gets a new id, and the module holding g_noalloc_scratch is loaded anew in it.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = (CtxGetCurrentFn)p;
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = (CtxGetIdFn)p;
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of g_noalloc_scratch, looked up with cudaGetSymbolAddress
// once per device (with that device current) and kept with the id of the
// context it was looked up in.  In host code the symbol itself is only a
// host-side stand-in, never a device address.  If the device's context has
// changed since (a reset), the address is looked up again: the old one
// belonged to the destroyed context.
void *scratch_address(int *err) {
  static std::mutex mu;
  static void *addr[64] = {nullptr};
  static unsigned long long ctx_of[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    *err = 1;
    return nullptr;
  }
  // the first runtime call above made the device's primary context current
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev] || ctx == 0 || ctx != ctx_of[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      *err = 2;
      addr[dev] = nullptr;
      return nullptr;
    }
    addr[dev] = p;
    ctx_of[dev] = ctx;
  }
  *err = 0;
  return addr[dev];
}

}  // namespace

using namespace mla;

extern "C" mla_status_t mla_decode_noalloc(const void *q, const void *cache, int64_t num_blocks,
                                           int32_t block_size, const int32_t *block_table,
                                           int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                           int32_t batch, int32_t num_heads, int32_t max_seq_len,
                                           float softmax_scale, void *out, float *lse,
                                           int32_t *dev_status, void *stream) {
  noalloc_fail(MLA_OK, "");
  if (batch > MLA_NOALLOC_MAX_BATCH)
    return noalloc_fail(MLA_ERR_INVALID_ARGUMENT,
                        "batch exceeds MLA_NOALLOC_MAX_BATCH (the fixed scratch holds the plan "
                        "for at most 8192 requests)");
  if (batch < 0 || num_heads != kHeads || block_size <= 0)
    return noalloc_fail(batch < 0 || block_size <= 0 ? MLA_ERR_INVALID_ARGUMENT
                                                      : MLA_ERR_UNSUPPORTED,
                        "batch >= 0, num_heads == 128 and block_size > 0 are required");
  if (batch == 0) return MLA_OK;
  // Ranges of the split plan: one per co-resident CTA pair, as many as the
  // fixed scratch holds.
  const int pairs = tc_max_pairs();
  if (pairs <= 0) return noalloc_fail(MLA_ERR_CUDA, "cannot query the current device");
  int ranges = pairs;
  while (ranges > 1 && workspace_layout(batch, kHeads, ranges).total > MLA_NOALLOC_SCRATCH_BYTES)
    --ranges;
  if (workspace_layout(batch, kHeads, ranges).total > MLA_NOALLOC_SCRATCH_BYTES)
    return noalloc_fail(MLA_ERR_INVALID_ARGUMENT, "batch too large for the fixed scratch");
  if (!q || !cache || !block_table || !seq_lens || !out)
    return noalloc_fail(MLA_ERR_INVALID_ARGUMENT, "null pointer argument");
  if (((uintptr_t)q | (uintptr_t)cache | (uintptr_t)out) % 16)
    return noalloc_fail(MLA_ERR_INVALID_ARGUMENT, "q, cache and out must be 16-byte aligned");
  if (((uintptr_t)block_table | (uintptr_t)seq_lens | (uintptr_t)lse) % 4)
    return noalloc_fail(MLA_ERR_INVALID_ARGUMENT, "block_table, seq_lens, lse: 4-byte alignment");
  if (block_size != 16 && block_size != 32 && block_size != 64 && block_size != 128 &&
      block_size != 256)
    return noalloc_fail(MLA_ERR_UNSUPPORTED, "block_size not in {16,32,64,128,256}");
  if (num_blocks <= 0 || num_blocks > (int64_t)INT32_MAX || max_blocks_per_seq <= 0 ||
      !plan_fits(batch, max_blocks_per_seq, block_size, tc_unit_tokens()) || max_seq_len < 0 ||
      (int64_t)max_seq_len > (int64_t)max_blocks_per_seq * block_size)
    return noalloc_fail(MLA_ERR_INVALID_ARGUMENT, "bad num_blocks, table width or max_seq_len");
  if (!(softmax_scale > 0.f) || softmax_scale == INFINITY)
    return noalloc_fail(MLA_ERR_INVALID_ARGUMENT, "softmax_scale must be positive and finite");
  int err = 0;
  void *ws = scratch_address(&err);
  if (!ws) return noalloc_fail(MLA_ERR_CUDA, "cudaGetSymbolAddress of the scratch array failed");
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = launch_plan(seq_lens, block_table, num_blocks, batch, tc_unit_tokens(),
                              max_blocks_per_seq, block_size, ranges, ws, num_heads, dev_status,
                              st);
  if (e == cudaSuccess)
    e = launch_decode_tc(q, cache, num_blocks, block_size, block_table, max_blocks_per_seq, batch,
                         softmax_scale, out, lse, ws, ranges, dev_status, st);
  // the decode above is not a programmatic dependent, so its combine is one
  if (e == cudaSuccess) e = launch_plan_combine(ws, batch, num_heads, ranges, out, lse, st, true);
  if (e != cudaSuccess) return noalloc_fail(MLA_ERR_CUDA, cudaGetErrorString(e));
  return MLA_OK;
}
