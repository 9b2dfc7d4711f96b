// C-ABI entry points of libmla: argument checks, workspace sizing, launches.
// Every public function validates on the host before launching anything and
// returns an mla_status_t; details of a failure go to a thread-local string.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <string>

#include "common.cuh"
#include "trace.h"

namespace mla {
cudaError_t launch_cache_append(const void *kv_new, const int64_t *slots, int64_t num_tokens,
                                void *cache, int64_t num_slots, int32_t *dev_status,
                                cudaStream_t stream);
cudaError_t launch_cache_append_fp8(const void *kv_new, const int64_t *slots, int64_t num_tokens,
                                    void *cache, int64_t num_slots, float inv_scale,
                                    int32_t *dev_status, cudaStream_t stream);
cudaError_t launch_plan(const int32_t *seq_lens, const int32_t *block_table, int64_t num_blocks,
                        int32_t batch, int32_t unit_tokens, int32_t max_blocks_per_seq,
                        int32_t block_size, int32_t max_ranges, void *ws, int32_t heads,
                        int32_t *dev_status, cudaStream_t stream);
cudaError_t launch_plan_combine(void *ws, int32_t batch, int32_t heads, int32_t max_ranges,
                                void *out, float *lse, cudaStream_t stream, bool early);
cudaError_t launch_offsets_combine(const float *o_part, const float *lse_part,
                                   const int32_t *offsets, int32_t batch, int32_t heads, void *out,
                                   float *lse, cudaStream_t stream);
cudaError_t launch_wait_selftest(int32_t *dev_status, uint64_t budget_ns, uint64_t *elapsed_ns,
                                 cudaStream_t stream);
int tc_unit_tokens();
int tc_max_pairs();
int tp_max_heads();
int tp_max_ranges();
cudaError_t launch_decode_tp(const void *q, const void *cache, int64_t num_blocks,
                             int32_t block_size, const int32_t *block_table,
                             int32_t max_blocks_per_seq, int32_t batch, int32_t heads,
                             float softmax_scale, void *out, float *lse, void *ws,
                             int32_t max_ranges, int32_t *dev_status, cudaStream_t stream);
cudaError_t launch_tp_combine(void *ws, int32_t batch, int32_t heads, int32_t max_ranges,
                              void *out, float *lse, cudaStream_t stream);
cudaError_t launch_decode_tc(const void *q, const void *cache, int64_t num_blocks, int32_t block_size,
                             const int32_t *block_table, int32_t max_blocks_per_seq, int32_t batch,
                             float softmax_scale, void *out, float *lse, void *ws,
                             int32_t max_ranges, int32_t *dev_status, cudaStream_t stream,
                             const void *kv_new = nullptr, bool fp8 = false, float kv_scale = 1.f,
                             bool early_launch = false);

namespace {

thread_local std::string g_detail;

mla_status_t fail(mla_status_t s, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_detail = buf;
  return s;
}

mla_status_t cuda_fail(cudaError_t e, const char *what) {
  return fail(MLA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Ranges of the plan: one per co-resident CTA pair of the tensor-core kernel.
int max_ranges_current() { return tc_max_pairs(); }

// A tensor-parallel rank's few heads (1 to 32) run on their own kernel
// (decode_tp.cu), whose plan has one range per SM.
bool few_heads(int32_t num_heads) { return num_heads >= 1 && num_heads <= tp_max_heads(); }

// The 128-head bf16 decode is launched as a programmatic dependent (its setup
// may overlap the previous kernel's tail; see decode_tc.cu) when the split
// combine of the same batch, which releases its dependents at entry, runs in
// one wave of 128-thread blocks: early decode CTAs would otherwise hold SMs
// that the combine's later waves need (measured slower on 256 requests).
// The FP8 decode measured slower launched early and is not.
//
// The split combine is launched as a programmatic dependent of the decode
// when that decode was not launched early itself (a larger batch, or an FP8
// cache): its blocks then take the SMs that decode CTAs free and wait there
// for the whole decode.  After an early-launched decode that was slower
// (config 3: 2.088 against 2.042 ms), likely because the combine's one wave
// crowded onto the first SMs freed.
bool decode_launches_early(int32_t batch) {
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return false;
  const int64_t r = max_ranges_current();
  const int64_t lanes = (int64_t)batch * 8 <= r ? 16 : ((int64_t)batch * 4 <= r ? 4 : 1);
  return (int64_t)batch * (kVDim / 16) * lanes <= 16 * (int64_t)sms;
}

// 33 to 127 heads: the workspace holds q padded to 128 heads and the padded
// output and lse, behind the plan and partials.  The pad heads hold whatever the workspace held:
// every head is an independent row of the kernel's work and of the merge, and
// only the caller's heads are copied out.
struct Padded {
  size_t q, out, lse, total;
};
Padded padded_layout(int32_t batch) {
  Padded p;
  p.q = 0;
  p.out = align256(p.q + (size_t)batch * kHeads * kRow * 2);
  p.lse = align256(p.out + (size_t)batch * kHeads * kVDim * 2);
  p.total = align256(p.lse + (size_t)batch * kHeads * 4);
  return p;
}

// The FP8 entry points work on the tensor-core kernel's own 128 heads only
mla_status_t need_all_heads(int32_t num_heads) {
  if (num_heads != kHeads)
    return fail(MLA_ERR_UNSUPPORTED, "num_heads %d: this entry point needs %d", num_heads, kHeads);
  return MLA_OK;
}

bool kv_scale_ok(float kv_scale) { return std::isfinite(kv_scale) && kv_scale > 0.f; }

bool block_size_ok(int32_t bs) { return bs == 16 || bs == 32 || bs == 64 || bs == 128 || bs == 256; }

mla_status_t check_decode_args(const void *q, const void *cache, int64_t num_blocks,
                               int32_t block_size, const int32_t *block_table,
                               int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t batch,
                               int32_t num_heads, int32_t max_seq_len, float softmax_scale,
                               void *out, float *lse, void *workspace, size_t workspace_bytes) {
  if (batch < 0) return fail(MLA_ERR_INVALID_ARGUMENT, "batch %d < 0", batch);
  if (num_heads < 1 || num_heads > kHeads)
    return fail(MLA_ERR_UNSUPPORTED, "num_heads %d: 1 to %d are supported", num_heads, kHeads);
  if (block_size <= 0) return fail(MLA_ERR_INVALID_ARGUMENT, "block_size %d <= 0", block_size);
  if (!block_size_ok(block_size))
    return fail(MLA_ERR_UNSUPPORTED, "block_size %d not in {16,32,64,128,256}", block_size);
  if (batch == 0) return MLA_OK;
  if (!q || !cache || !block_table || !seq_lens || !out || !workspace)
    return fail(MLA_ERR_INVALID_ARGUMENT, "null pointer argument");
  if (!aligned(q, 16) || !aligned(cache, 16) || !aligned(out, 16))
    return fail(MLA_ERR_INVALID_ARGUMENT, "q, cache and out must be 16-byte aligned");
  if (!aligned(block_table, 4) || !aligned(seq_lens, 4) || (lse && !aligned(lse, 4)))
    return fail(MLA_ERR_INVALID_ARGUMENT, "block_table, seq_lens, lse must be 4-byte aligned");
  if (!aligned(workspace, 256))
    return fail(MLA_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");
  if (num_blocks <= 0 || num_blocks > (int64_t)INT32_MAX)
    return fail(MLA_ERR_INVALID_ARGUMENT, "num_blocks %lld out of range", (long long)num_blocks);
  if (max_blocks_per_seq <= 0)
    return fail(MLA_ERR_INVALID_ARGUMENT, "max_blocks_per_seq %d <= 0", max_blocks_per_seq);
  if (!plan_fits(batch, max_blocks_per_seq, block_size, tc_unit_tokens()))
    return fail(MLA_ERR_INVALID_ARGUMENT, "batch * max_blocks_per_seq * block_size too large");
  if (max_seq_len < 0 || (int64_t)max_seq_len > (int64_t)max_blocks_per_seq * block_size)
    return fail(MLA_ERR_INVALID_ARGUMENT, "max_seq_len %d outside [0, %lld]", max_seq_len,
                (long long)max_blocks_per_seq * block_size);
  if (!std::isfinite(softmax_scale) || !(softmax_scale > 0.f))
    return fail(MLA_ERR_INVALID_ARGUMENT, "softmax_scale must be positive and finite");
  const size_t need = mla_decode_workspace_size(batch, num_heads);
  if (need == 0) return fail(MLA_ERR_CUDA, "cannot query the current device");
  if (workspace_bytes < need)
    return fail(MLA_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %zu needed", workspace_bytes,
                need);
  return MLA_OK;
}

}  // namespace

// Failure reporting for the fixed-scratch entry point (noalloc.cu).
mla_status_t noalloc_fail(mla_status_t s, const char *msg) { return fail(s, "%s", msg); }

// The thread's error detail (read by mla_last_error_detail), for the host-only
// entry points of placement.cu.
void set_error_detail(const char *msg) { g_detail = msg ? msg : ""; }

}  // namespace mla

using namespace mla;

extern "C" {

const char *mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARGUMENT: return "MLA_ERR_INVALID_ARGUMENT";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_WORKSPACE_TOO_SMALL: return "MLA_ERR_WORKSPACE_TOO_SMALL";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_DEVICE_RANGE: return "MLA_ERR_DEVICE_RANGE";
    case MLA_ERR_DEVICE_TIMEOUT: return "MLA_ERR_DEVICE_TIMEOUT";
    case MLA_ERR_DEVICE_PLAN: return "MLA_ERR_DEVICE_PLAN";
    default: return "MLA_ERR_UNKNOWN";
  }
}

const char *mla_last_error_detail(void) { return g_detail.c_str(); }

int mla_abi_version(void) { return MLA_ABI_VERSION; }

mla_status_t mla_cache_append(const void *kv_new, const int64_t *slot_mapping, int64_t num_tokens,
                              void *cache, int64_t num_blocks, int32_t block_size,
                              int32_t *dev_status, void *stream) {
  TraceRange trace_range("mla_cache_append");
  g_detail.clear();
  if (num_tokens < 0) return fail(MLA_ERR_INVALID_ARGUMENT, "num_tokens < 0");
  if (block_size <= 0) return fail(MLA_ERR_INVALID_ARGUMENT, "block_size %d <= 0", block_size);
  if (num_blocks <= 0) return fail(MLA_ERR_INVALID_ARGUMENT, "num_blocks <= 0");
  if (num_tokens == 0) return MLA_OK;
  if (!kv_new || !slot_mapping || !cache) return fail(MLA_ERR_INVALID_ARGUMENT, "null pointer");
  if (!aligned(kv_new, 16) || !aligned(cache, 16) || !aligned(slot_mapping, 8))
    return fail(MLA_ERR_INVALID_ARGUMENT, "kv_new/cache must be 16-byte, slot_mapping 8-byte aligned");
  cudaError_t e = launch_cache_append(kv_new, slot_mapping, num_tokens, cache,
                                      num_blocks * (int64_t)block_size, dev_status,
                                      (cudaStream_t)stream);
  return e == cudaSuccess ? MLA_OK : cuda_fail(e, "mla_cache_append launch");
}

size_t mla_decode_workspace_size(int32_t batch, int32_t num_heads) {
  if (batch < 0 || num_heads <= 0 || num_heads > kHeads) return 0;
  if (few_heads(num_heads)) {
    const int ranges = tp_max_ranges();
    return ranges <= 0 ? 0 : workspace_layout(batch, num_heads, ranges).total;
  }
  const int ranges = max_ranges_current();
  if (ranges <= 0) return 0;
  const size_t plan = workspace_layout(batch, kHeads, ranges).total;
  return num_heads == kHeads ? plan : plan + padded_layout(batch).total;
}

mla_status_t mla_decode_plan(const int32_t *seq_lens, const int32_t *block_table, int32_t batch,
                             int32_t num_heads, int32_t max_blocks_per_seq, int32_t block_size,
                             int64_t num_blocks, void *workspace, size_t workspace_bytes,
                             int32_t *dev_status, void *stream) {
  TraceRange trace_range("mla_decode_plan");
  g_detail.clear();
  if (batch < 0) return fail(MLA_ERR_INVALID_ARGUMENT, "batch < 0");
  if (num_heads < 1 || num_heads > kHeads)
    return fail(MLA_ERR_UNSUPPORTED, "num_heads %d: 1 to %d are supported", num_heads, kHeads);
  if (!block_size_ok(block_size)) return fail(MLA_ERR_UNSUPPORTED, "block_size %d", block_size);
  if (batch == 0) return MLA_OK;
  if (!seq_lens || !workspace) return fail(MLA_ERR_INVALID_ARGUMENT, "null pointer");
  if (!aligned(workspace, 256)) return fail(MLA_ERR_INVALID_ARGUMENT, "workspace alignment");
  if (max_blocks_per_seq <= 0) return fail(MLA_ERR_INVALID_ARGUMENT, "max_blocks_per_seq <= 0");
  if (!plan_fits(batch, max_blocks_per_seq, block_size, tc_unit_tokens()))
    return fail(MLA_ERR_INVALID_ARGUMENT, "batch * max_blocks_per_seq * block_size too large");
  const size_t need = mla_decode_workspace_size(batch, num_heads);
  if (need == 0) return fail(MLA_ERR_CUDA, "cannot query the current device");
  if (workspace_bytes < need)
    return fail(MLA_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu", workspace_bytes, need);
  if (block_table && num_blocks <= 0)
    return fail(MLA_ERR_INVALID_ARGUMENT, "num_blocks must be > 0 with a block table");
  const bool few = few_heads(num_heads);
  cudaError_t e = launch_plan(seq_lens, block_table, num_blocks, batch, tc_unit_tokens(),
                              max_blocks_per_seq, block_size,
                              few ? tp_max_ranges() : max_ranges_current(), workspace,
                              few ? num_heads : kHeads, dev_status, (cudaStream_t)stream);
  return e == cudaSuccess ? MLA_OK : cuda_fail(e, "plan launch");
}

mla_status_t mla_decode_partial(const void *q, void *cache, const void *kv_new,
                                int64_t num_blocks, int32_t block_size,
                                const int32_t *block_table, int32_t max_blocks_per_seq,
                                const int32_t *seq_lens, int32_t batch, int32_t num_heads,
                                int32_t max_seq_len, float softmax_scale, void *out, float *lse,
                                void *workspace, size_t workspace_bytes, int32_t *dev_status,
                                void *stream) {
  TraceRange trace_range("mla_decode_partial");
  g_detail.clear();
  const bool few = few_heads(num_heads);
  if (!few && num_heads != kHeads)
    return fail(MLA_ERR_UNSUPPORTED, "num_heads %d: this entry point takes 1 to %d or %d",
                num_heads, tp_max_heads(), kHeads);
  if (few && kv_new)
    return fail(MLA_ERR_UNSUPPORTED, "the fused append needs %d heads", kHeads);
  mla_status_t s = check_decode_args(q, cache, num_blocks, block_size, block_table,
                                     max_blocks_per_seq, seq_lens, batch, num_heads, max_seq_len,
                                     softmax_scale, out, lse, workspace, workspace_bytes);
  if (s != MLA_OK || batch == 0) return s;
  if (kv_new && !aligned(kv_new, 16))
    return fail(MLA_ERR_INVALID_ARGUMENT, "kv_new must be 16-byte aligned");
  if (few) {
    cudaError_t e = launch_decode_tp(q, cache, num_blocks, block_size, block_table,
                                     max_blocks_per_seq, batch, num_heads, softmax_scale, out,
                                     lse, workspace, tp_max_ranges(), dev_status,
                                     (cudaStream_t)stream);
    return e == cudaSuccess ? MLA_OK : cuda_fail(e, "few-head decode launch");
  }
  cudaError_t e = launch_decode_tc(q, cache, num_blocks, block_size, block_table,
                                   max_blocks_per_seq, batch, softmax_scale, out, lse, workspace,
                                   max_ranges_current(), dev_status, (cudaStream_t)stream, kv_new,
                                   false, 1.f, decode_launches_early(batch));
  return e == cudaSuccess ? MLA_OK : cuda_fail(e, "decode launch");
}

mla_status_t mla_decode_append_planned(const void *q, void *cache, const void *kv_new,
                                       int64_t num_blocks, int32_t block_size,
                                       const int32_t *block_table, int32_t max_blocks_per_seq,
                                       const int32_t *seq_lens, int32_t batch, int32_t num_heads,
                                       int32_t max_seq_len, float softmax_scale, void *out,
                                       float *lse, void *workspace, size_t workspace_bytes,
                                       int32_t *dev_status, void *stream) {
  TraceRange trace_range("mla_decode_append_planned");
  if (!kv_new) {
    g_detail.clear();
    return fail(MLA_ERR_INVALID_ARGUMENT, "kv_new is null");
  }
  mla_status_t s = mla_decode_partial(q, cache, kv_new, num_blocks, block_size, block_table,
                                      max_blocks_per_seq, seq_lens, batch, num_heads, max_seq_len,
                                      softmax_scale, out, lse, workspace, workspace_bytes,
                                      dev_status, stream);
  if (s != MLA_OK || batch == 0) return s;
  return mla_combine_planned(workspace, workspace_bytes, batch, num_heads, out, lse, stream);
}

mla_status_t mla_combine_planned(void *workspace, size_t workspace_bytes, int32_t batch,
                                 int32_t num_heads, void *out, float *lse, void *stream) {
  TraceRange trace_range("mla_combine_planned");
  g_detail.clear();
  if (batch < 0) return fail(MLA_ERR_INVALID_ARGUMENT, "batch < 0");
  const bool few = few_heads(num_heads);
  if (!few && num_heads != kHeads)
    return fail(MLA_ERR_UNSUPPORTED, "num_heads %d: this entry point takes 1 to %d or %d",
                num_heads, tp_max_heads(), kHeads);
  if (batch == 0) return MLA_OK;
  if (!workspace || !out) return fail(MLA_ERR_INVALID_ARGUMENT, "null pointer");
  if (!aligned(workspace, 256) || !aligned(out, 16) || (lse && !aligned(lse, 4)))
    return fail(MLA_ERR_INVALID_ARGUMENT, "workspace / out / lse alignment");
  const size_t need = mla_decode_workspace_size(batch, num_heads);
  if (need == 0) return fail(MLA_ERR_CUDA, "cannot query the current device");
  if (workspace_bytes < need)
    return fail(MLA_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu", workspace_bytes, need);
  cudaError_t e =
      few ? launch_tp_combine(workspace, batch, num_heads, tp_max_ranges(), out, lse,
                              (cudaStream_t)stream)
          : launch_plan_combine(workspace, batch, num_heads, max_ranges_current(), out, lse,
                                (cudaStream_t)stream, !decode_launches_early(batch));
  return e == cudaSuccess ? MLA_OK : cuda_fail(e, "combine launch");
}

mla_status_t mla_decode_planned(const void *q, const void *cache, int64_t num_blocks,
                                int32_t block_size, const int32_t *block_table,
                                int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                int32_t batch, int32_t num_heads, int32_t max_seq_len,
                                float softmax_scale, void *out, float *lse, void *workspace,
                                size_t workspace_bytes, int32_t *dev_status, void *stream) {
  TraceRange trace_range("mla_decode_planned");
  if (num_heads != kHeads && !few_heads(num_heads)) {  // 33 to 127 heads, padded to 128
    g_detail.clear();
    mla_status_t st = check_decode_args(q, cache, num_blocks, block_size, block_table,
                                        max_blocks_per_seq, seq_lens, batch, num_heads,
                                        max_seq_len, softmax_scale, out, lse, workspace,
                                        workspace_bytes);
    if (st != MLA_OK || batch == 0) return st;
    const Padded pl = padded_layout(batch);
    char *pad = (char *)workspace + workspace_layout(batch, kHeads, max_ranges_current()).total;
    void *q_pad = pad + pl.q, *out_pad = pad + pl.out;
    float *lse_pad = (float *)(pad + pl.lse);
    const size_t qrow = (size_t)num_heads * kRow * 2, orow = (size_t)num_heads * kVDim * 2;
    cudaError_t e = cudaMemcpy2DAsync(q_pad, (size_t)kHeads * kRow * 2, q, qrow, qrow, batch,
                                      cudaMemcpyDeviceToDevice, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "q copy into the padded heads");
    st = mla_decode_partial(q_pad, const_cast<void *>(cache), nullptr, num_blocks, block_size,
                            block_table, max_blocks_per_seq, seq_lens, batch, kHeads, max_seq_len,
                            softmax_scale, out_pad, lse_pad, workspace, workspace_bytes,
                            dev_status, stream);
    if (st != MLA_OK) return st;
    st = mla_combine_planned(workspace, workspace_bytes, batch, kHeads, out_pad, lse_pad, stream);
    if (st != MLA_OK) return st;
    e = cudaMemcpy2DAsync(out, orow, out_pad, (size_t)kHeads * kVDim * 2, orow, batch,
                          cudaMemcpyDeviceToDevice, (cudaStream_t)stream);
    if (e == cudaSuccess && lse)
      e = cudaMemcpy2DAsync(lse, (size_t)num_heads * 4, lse_pad, (size_t)kHeads * 4,
                            (size_t)num_heads * 4, batch, cudaMemcpyDeviceToDevice,
                            (cudaStream_t)stream);
    return e == cudaSuccess ? MLA_OK : cuda_fail(e, "output copy from the padded heads");
  }
  mla_status_t s = mla_decode_partial(q, const_cast<void *>(cache), nullptr, num_blocks,
                                      block_size, block_table, max_blocks_per_seq, seq_lens,
                                      batch, num_heads, max_seq_len, softmax_scale, out, lse,
                                      workspace, workspace_bytes, dev_status, stream);
  if (s != MLA_OK || batch == 0) return s;
  return mla_combine_planned(workspace, workspace_bytes, batch, num_heads, out, lse, stream);
}

mla_status_t mla_decode(const void *q, const void *cache, int64_t num_blocks, int32_t block_size,
                        const int32_t *block_table, int32_t max_blocks_per_seq,
                        const int32_t *seq_lens, int32_t batch, int32_t num_heads,
                        int32_t max_seq_len, float softmax_scale, void *out, float *lse,
                        void *workspace, size_t workspace_bytes, int32_t *dev_status,
                        void *stream) {
  TraceRange trace_range("mla_decode");
  g_detail.clear();
  mla_status_t s = check_decode_args(q, cache, num_blocks, block_size, block_table,
                                     max_blocks_per_seq, seq_lens, batch, num_heads, max_seq_len,
                                     softmax_scale, out, lse, workspace, workspace_bytes);
  if (s != MLA_OK || batch == 0) return s;
  s = mla_decode_plan(seq_lens, block_table, batch, num_heads, max_blocks_per_seq, block_size,
                      num_blocks, workspace, workspace_bytes, dev_status, stream);
  if (s != MLA_OK) return s;
  return mla_decode_planned(q, cache, num_blocks, block_size, block_table, max_blocks_per_seq,
                            seq_lens, batch, num_heads, max_seq_len, softmax_scale, out, lse,
                            workspace, workspace_bytes, dev_status, stream);
}

mla_status_t mla_combine(const float *o_partial, const float *lse_partial,
                         const int32_t *split_offsets, int32_t batch, int32_t num_heads,
                         void *out, float *lse, void *stream) {
  TraceRange trace_range("mla_combine");
  g_detail.clear();
  if (batch < 0 || num_heads <= 0)
    return fail(MLA_ERR_INVALID_ARGUMENT, "batch %d, num_heads %d", batch, num_heads);
  if (batch == 0) return MLA_OK;
  if (!o_partial || !lse_partial || !split_offsets || !out)
    return fail(MLA_ERR_INVALID_ARGUMENT, "null pointer");
  if (!aligned(o_partial, 16) || !aligned(out, 16) || !aligned(lse_partial, 4))
    return fail(MLA_ERR_INVALID_ARGUMENT, "o_partial/out must be 16-byte aligned");
  if (num_heads > 65535) return fail(MLA_ERR_INVALID_ARGUMENT, "num_heads %d > 65535", num_heads);
  cudaError_t e = launch_offsets_combine(o_partial, lse_partial, split_offsets, batch, num_heads,
                                         out, lse, (cudaStream_t)stream);
  return e == cudaSuccess ? MLA_OK : cuda_fail(e, "combine launch");
}

mla_status_t mla_cache_append_fp8(const void *kv_new, const int64_t *slot_mapping,
                                  int64_t num_tokens, void *cache8, int64_t num_blocks,
                                  int32_t block_size, float kv_scale, int32_t *dev_status,
                                  void *stream) {
  TraceRange trace_range("mla_cache_append_fp8");
  g_detail.clear();
  if (num_tokens < 0) return fail(MLA_ERR_INVALID_ARGUMENT, "num_tokens < 0");
  if (block_size <= 0) return fail(MLA_ERR_INVALID_ARGUMENT, "block_size %d <= 0", block_size);
  if (num_blocks <= 0) return fail(MLA_ERR_INVALID_ARGUMENT, "num_blocks <= 0");
  if (!kv_scale_ok(kv_scale))
    return fail(MLA_ERR_INVALID_ARGUMENT, "kv_scale must be positive and finite");
  if (num_tokens == 0) return MLA_OK;
  if (!kv_new || !slot_mapping || !cache8) return fail(MLA_ERR_INVALID_ARGUMENT, "null pointer");
  if (!aligned(kv_new, 16) || !aligned(cache8, 16) || !aligned(slot_mapping, 8))
    return fail(MLA_ERR_INVALID_ARGUMENT,
                "kv_new/cache8 must be 16-byte, slot_mapping 8-byte aligned");
  cudaError_t e = launch_cache_append_fp8(kv_new, slot_mapping, num_tokens, cache8,
                                          num_blocks * (int64_t)block_size, 1.f / kv_scale,
                                          dev_status, (cudaStream_t)stream);
  return e == cudaSuccess ? MLA_OK : cuda_fail(e, "mla_cache_append_fp8 launch");
}

mla_status_t mla_decode_fp8_planned(const void *q, void *cache8, const void *kv_new,
                                    int64_t num_blocks, int32_t block_size,
                                    const int32_t *block_table, int32_t max_blocks_per_seq,
                                    const int32_t *seq_lens, int32_t batch, int32_t num_heads,
                                    int32_t max_seq_len, float softmax_scale, float kv_scale,
                                    void *out, float *lse, void *workspace, size_t workspace_bytes,
                                    int32_t *dev_status, void *stream) {
  TraceRange trace_range("mla_decode_fp8_planned");
  g_detail.clear();
  if (need_all_heads(num_heads) != MLA_OK) return MLA_ERR_UNSUPPORTED;
  mla_status_t s = check_decode_args(q, cache8, num_blocks, block_size, block_table,
                                     max_blocks_per_seq, seq_lens, batch, num_heads, max_seq_len,
                                     softmax_scale, out, lse, workspace, workspace_bytes);
  if (s != MLA_OK) return s;
  if (!kv_scale_ok(kv_scale))
    return fail(MLA_ERR_INVALID_ARGUMENT, "kv_scale must be positive and finite");
  if (batch == 0) return MLA_OK;
  if (kv_new && !aligned(kv_new, 16))
    return fail(MLA_ERR_INVALID_ARGUMENT, "kv_new must be 16-byte aligned");
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = launch_decode_tc(q, cache8, num_blocks, block_size, block_table,
                                   max_blocks_per_seq, batch, softmax_scale, out, lse, workspace,
                                   max_ranges_current(), dev_status, st, kv_new, true, kv_scale);
  if (e != cudaSuccess) return cuda_fail(e, "FP8 decode launch");
  e = launch_plan_combine(workspace, batch, num_heads, max_ranges_current(), out, lse, st, true);
  return e == cudaSuccess ? MLA_OK : cuda_fail(e, "combine launch");
}

mla_status_t mla_decode_fp8(const void *q, const void *cache8, int64_t num_blocks,
                            int32_t block_size, const int32_t *block_table,
                            int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t batch,
                            int32_t num_heads, int32_t max_seq_len, float softmax_scale,
                            float kv_scale, void *out, float *lse, void *workspace,
                            size_t workspace_bytes, int32_t *dev_status, void *stream) {
  TraceRange trace_range("mla_decode_fp8");
  g_detail.clear();
  if (need_all_heads(num_heads) != MLA_OK) return MLA_ERR_UNSUPPORTED;
  mla_status_t s = check_decode_args(q, cache8, num_blocks, block_size, block_table,
                                     max_blocks_per_seq, seq_lens, batch, num_heads, max_seq_len,
                                     softmax_scale, out, lse, workspace, workspace_bytes);
  if (s != MLA_OK) return s;
  if (!kv_scale_ok(kv_scale))
    return fail(MLA_ERR_INVALID_ARGUMENT, "kv_scale must be positive and finite");
  if (batch == 0) return MLA_OK;
  s = mla_decode_plan(seq_lens, block_table, batch, num_heads, max_blocks_per_seq, block_size,
                      num_blocks, workspace, workspace_bytes, dev_status, stream);
  if (s != MLA_OK) return s;
  return mla_decode_fp8_planned(q, const_cast<void *>(cache8), nullptr, num_blocks, block_size,
                                block_table, max_blocks_per_seq, seq_lens, batch, num_heads,
                                max_seq_len, softmax_scale, kv_scale, out, lse, workspace,
                                workspace_bytes, dev_status, stream);
}

mla_status_t mla_selftest_wait_timeout(uint64_t budget_ns, int32_t *dev_status,
                                       uint64_t *elapsed_ns, void *stream) {
  TraceRange trace_range("mla_selftest_wait_timeout");
  g_detail.clear();
  if (budget_ns < 1000 || budget_ns > 1000000000ull)
    return fail(MLA_ERR_INVALID_ARGUMENT, "budget_ns %llu: 1 us to 1 s",
                (unsigned long long)budget_ns);
  if (!dev_status || !elapsed_ns) return fail(MLA_ERR_INVALID_ARGUMENT, "null pointer");
  if (!aligned(dev_status, 4) || !aligned(elapsed_ns, 8))
    return fail(MLA_ERR_INVALID_ARGUMENT, "dev_status / elapsed_ns alignment");
  cudaError_t e = launch_wait_selftest(dev_status, budget_ns, elapsed_ns, (cudaStream_t)stream);
  return e == cudaSuccess ? MLA_OK : cuda_fail(e, "self-test launch");
}

}  // extern "C"
