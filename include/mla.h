/*
 * libmla — MLA latent-cache decode for one data-parallel-attention rank on a
 * GB300 (sm_103a).  C ABI: plain pointers and sizes, no framework types.
 *
 * The operation (absorbed-form Multi-head Latent Attention decode):
 *   Each cached token holds ONE 576-wide latent row shared by all heads:
 *   elements 0..511 are kv_c (kv_lora_rank = 512) and 512..575 the MQA-style
 *   k_rope (64 dims shared by every head), stored per layer as [NB, BS, 576]
 *   [MLA 的 TP 切分：为什么 8 张 GPU 存了同一份 KV cache (10100.com), section 2.2
 *   "三个事实" and section 3.1 (MLAAttentionSpec: num_kv_heads = 1,
 *   head_size = 576; per-layer cache [NB, BS, 576])].
 *   In decode the engine runs the absorbed form: every head's query is already
 *   projected into the latent space (q_nope . W_UK -> 512 dims, plus 64 rope
 *   dims) and attends over the shared latent directly
 *   [dp-attention-expert-parallel-mla-kv-replication (inferenceinterviews.com),
 *   "A strong answer"].  The value is the 512-dim kv_c itself
 *   (v_head_dim = kv_lora_rank) [DP 与 DPA 的区别：SGLang 并行部署与路由
 *   (chengxuchu.com), "MLA：KV 是一份共享 latent"].  For request b with context
 *   length L and head h:
 *       s_t  = softmax_scale * sum_{d<576} q[b,h,d] * row_t[d]
 *       out[b,h,j] = sum_t softmax(s)_t * row_t[j]          (j < 512)
 *       lse[b,h]   = log sum_t exp(s_t)                     (natural log)
 *   where row_t = cache[block_table[b][t / BS]][t % BS].
 *   With data-parallel attention a rank owns its requests, their cache and the
 *   full attention weights, so this step needs no communication between GPUs
 *   [dp-attention-expert-parallel-mla-kv-replication, "The fix"]; a rank with no
 *   requests still runs the step with an empty batch ["What it costs"], which
 *   here is batch = 0, a valid no-op.
 *
 * Conventions shared by every entry point
 *   - Device pointers are CUDA device (or managed) memory of the current
 *     device; host pointers are named *_host.  The caller owns every buffer.
 *     The library allocates and frees nothing, never synchronises, and launches
 *     only on the caller's stream (a cudaStream_t passed as void*; NULL = the
 *     legacy default stream).
 *   - Tensors are dense, row-major, with the shapes given.  bf16 = IEEE
 *     bfloat16 stored as 16-bit values.  Device pointers to bf16/fp32 data
 *     must be 16-byte aligned.
 *   - Arguments are checked on the host before any launch; a failed check
 *     returns a status and launches nothing.  mla_last_error_detail() then
 *     describes it (thread-local string).
 *   - Faults the host cannot see (a block-table entry or slot outside the
 *     pool, a sequence longer than its table) are reported by the kernels into
 *     *dev_status (optional, device int32, first error wins; 0 = none): the
 *     kernels never trap.  Read it after synchronising the stream.  Results of
 *     a request touched by such a fault are unspecified.
 *   - Every bounded wait inside a kernel gives up after a fixed time budget
 *     and reports MLA_ERR_DEVICE_TIMEOUT in *dev_status instead of hanging.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_ABI_VERSION 4
#define MLA_ROW_DIM 576       /* 512 kv_c + 64 k_rope per cached token */
#define MLA_KV_LORA_RANK 512  /* value / output width */
#define MLA_ROPE_DIM 64
#define MLA_NUM_HEADS 128     /* heads per request the decode supports */

typedef enum mla_status {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARGUMENT = 1,    /* host-side check failed, nothing launched */
  MLA_ERR_UNSUPPORTED = 2,         /* valid but not supported (e.g. num_heads != 128) */
  MLA_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes < mla_decode_workspace_size() */
  MLA_ERR_CUDA = 4,                /* a CUDA runtime call or launch failed */
  MLA_ERR_DEVICE_RANGE = 5,        /* device-seen: bad block id, slot or length */
  MLA_ERR_DEVICE_TIMEOUT = 6,      /* device-seen: a bounded wait expired */
  MLA_ERR_DEVICE_PLAN = 7          /* device-seen: the workspace holds no plan for these
                                      arguments (batch, heads, page size, table width);
                                      nothing was decoded */
} mla_status_t;

/* Name of a status code ("MLA_OK", ...); never NULL. */
const char *mla_status_string(int status);

/* Detail of the last failed call on this host thread ("" if none). */
const char *mla_last_error_detail(void);

/* MLA_ABI_VERSION of the loaded library. */
int mla_abi_version(void);

/*
 * mla_cache_append — store each new token's 576-wide latent row into its slot.
 *
 * Defined by: the per-token output of kv_a_proj_with_mqa is one 512 + 64 = 576
 * wide row, replicated rather than split by head, and it is what the MLA cache
 * stores [MLA 的 TP 切分 (10100.com), section 2.2 and 3.1].
 *
 *   kv_new        bf16 [num_tokens, 576]  rows to store (copied bit-exactly).
 *   slot_mapping  int64 [num_tokens]      slot = block * block_size + row;
 *                                         -1 = skip this token.
 *   cache         bf16 [num_blocks, block_size, 576], updated in place.
 * num_tokens = 0 is a no-op.  A slot outside [-1, num_blocks*block_size) is
 * skipped and reported as MLA_ERR_DEVICE_RANGE in *dev_status.  Two tokens
 * with the same slot race (either row may win).  block_size >= 1.
 */
mla_status_t mla_cache_append(const void *kv_new, const int64_t *slot_mapping,
                              int64_t num_tokens, void *cache, int64_t num_blocks,
                              int32_t block_size, int32_t *dev_status, void *stream);

/*
 * mla_decode_workspace_size — bytes of scratch mla_decode needs on the
 * current device for `batch` requests of `num_heads` heads.  The workspace
 * holds the split plan (units of the token partition, per request) and the
 * partial results of requests that are split across CTAs (each range's
 * normalised output in bf16 with its fp32 log-sum-exp).  It depends on
 * neither the context lengths nor the page size: the plan has at most one
 * range per SM pair of the current device (one per SM for 1 to 32 heads)
 * and each range leaves at most two partials, whatever the lengths.  Returns
 * 0 for batch < 0, num_heads outside [1, 128] or no current device.
 */
size_t mla_decode_workspace_size(int32_t batch, int32_t num_heads);

/*
 * mla_decode_plan — compute the split-KV plan for these sequence lengths
 * into the workspace (one small kernel).  The plan depends on seq_lens,
 * batch, max_blocks_per_seq, block_size and — when block_table is given
 * (device int32 [batch, max_blocks_per_seq], nullable) — on the table too: it
 * then records where each worker's first tile lies in the cache (num_blocks
 * is the pool size, > 0), so the decode starts loading without a table
 * lookup; re-plan when any of them changes.  A caller decoding many layers
 * of one step with the same lengths and table plans once and then calls
 * mla_decode_planned per layer.  Lengths are read on the device; a length
 * outside [0, max_blocks_per_seq * block_size] is clamped and reported as
 * MLA_ERR_DEVICE_RANGE.
 */
mla_status_t mla_decode_plan(const int32_t *seq_lens, const int32_t *block_table, int32_t batch,
                             int32_t num_heads, int32_t max_blocks_per_seq, int32_t block_size,
                             int64_t num_blocks, void *workspace, size_t workspace_bytes,
                             int32_t *dev_status, void *stream);

/*
 * mla_decode — absorbed-form MLA decode (the equation at the top of this file).
 * Runs mla_decode_plan and then mla_decode_planned.
 *
 *   q             bf16 [batch, num_heads, 576]  absorbed queries (512 latent
 *                 dims from q_nope . W_UK, then 64 already-rotated rope dims).
 *   cache         bf16 [num_blocks, block_size, 576] this layer's latent cache.
 *   block_table   int32 [batch, max_blocks_per_seq]; entry i of request b is
 *                 the physical block of tokens [i*BS, (i+1)*BS).  Only the
 *                 first ceil(seq_lens[b] / BS) entries are read.
 *   seq_lens      int32 [batch] (device) context lengths; 0 gives out = 0 and
 *                 lse = -inf for that request.
 *   max_seq_len   host upper bound of seq_lens (checked against the table).
 *   softmax_scale multiplies q . row (e.g. 1/sqrt(192) for 128 + 64 dim heads);
 *                 positive and finite, else MLA_ERR_INVALID_ARGUMENT.
 *   out           bf16 [batch, num_heads, 512] (written).
 *   lse           fp32 [batch, num_heads] natural-log sum-exp, or NULL.
 *   workspace     device scratch of >= mla_decode_workspace_size(batch,
 *                 num_heads) bytes, 256-byte aligned; its contents on entry
 *                 do not matter (the plan rewrites everything the decode
 *                 reads).  Calls sharing one workspace must not overlap on
 *                 the GPU.
 * Heads: 1 <= num_heads <= 128.  128 heads run on the tensor-core kernel
 * whose CTA pairs split the output dims; 1 to 32 heads — a tensor-parallel
 * rank's share, e.g. 16 at TP = 8 [dp-attention-expert-parallel-mla-kv-
 * replication (inferenceinterviews.com), "A strong answer"] — run on a
 * kernel of their own, which computes the transposed products (tokens and
 * value dims in the MMA's M, heads in N) with one CTA per SM; 33 to 127 are
 * padded to 128 inside the workspace (mla_decode and mla_decode_planned
 * only).  mla_decode_workspace_size(batch, num_heads) sizes the workspace
 * for the path num_heads takes, and mla_decode_plan must be given the same
 * num_heads as the decode that uses its plan.
 * Requirements: block_size in {16, 32, 64, 128, 256};
 * max_seq_len <= max_blocks_per_seq * block_size <= 2^30; batch *
 * ceil(max_blocks_per_seq * block_size / 64) < 2^31 (the plan counts 64-token
 * units in int32); batch >= 0 (0 = no-op).  Else MLA_ERR_INVALID_ARGUMENT.
 * Rows the plan does not cover (tails past seq_len, unused blocks) are never
 * read, whatever they hold.
 * Launch order: every launch is ordered after the previous work on `stream`
 * as usual.  Some are programmatic dependents of the kernel before them (they
 * set up while it ends and wait for it to complete before touching memory),
 * and the 128-head decode releases its own programmatic dependents once its
 * CTAs have requested their last tile, before its outputs are written.  A
 * caller's kernel launched after these calls with programmatic stream
 * serialization must therefore wait for the grid before it reads their
 * outputs (griddepcontrol.wait), as the library's own kernels do; kernels
 * launched without that attribute are unaffected.
 */
mla_status_t mla_decode(const void *q, const void *cache, int64_t num_blocks, int32_t block_size,
                        const int32_t *block_table, int32_t max_blocks_per_seq,
                        const int32_t *seq_lens, int32_t batch, int32_t num_heads,
                        int32_t max_seq_len, float softmax_scale, void *out, float *lse,
                        void *workspace, size_t workspace_bytes, int32_t *dev_status,
                        void *stream);

/*
 * mla_decode_planned — mla_decode using the plan already in `workspace`
 * (from mla_decode_plan with the same seq_lens, batch, num_heads, block_size,
 * max_blocks_per_seq and, if it was given one, block table).  Same arguments
 * and results as mla_decode.  The planner stamps every segment record with
 * the arguments it was made for (batch, split ranges, page size, table
 * width) and the decode checks each record against its own, and against the
 * bounds of the request, table and workspace, before using it: a plan made
 * for other arguments is reported as MLA_ERR_DEVICE_PLAN in *dev_status and
 * out / lse are then unspecified; nothing is read or written out of place,
 * whatever the workspace holds.
 */
mla_status_t mla_decode_planned(const void *q, const void *cache, int64_t num_blocks,
                                int32_t block_size, const int32_t *block_table,
                                int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                int32_t batch, int32_t num_heads, int32_t max_seq_len,
                                float softmax_scale, void *out, float *lse, void *workspace,
                                size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * mla_decode_partial / mla_combine_planned — the two launches of
 * mla_decode_planned (and of mla_decode_append_planned), for callers that want
 * to place or time them apart.  mla_decode_partial runs the decode kernel over
 * the plan's token ranges: requests that lie in one range get their out (and
 * lse) written; requests spread over several ranges leave one partial result
 * per range in the workspace (its normalised output in bf16 and its fp32
 * log-sum-exp; the merge accumulates in fp32).  With kv_new non-null it first stores
 * each request's new row as mla_decode_append_planned does (the cache is
 * written then; with kv_new NULL it is only read).  mla_combine_planned then
 * merges the partials into out / lse (requests that were not split are left
 * as they are).  Same arguments and requirements as mla_decode_planned, with
 * num_heads 128 or 1 to 32 (else MLA_ERR_UNSUPPORTED); kv_new needs 128
 * heads.  The workspace must not be touched between the two calls.
 */
mla_status_t mla_decode_partial(const void *q, void *cache, const void *kv_new,
                                int64_t num_blocks, int32_t block_size,
                                const int32_t *block_table, int32_t max_blocks_per_seq,
                                const int32_t *seq_lens, int32_t batch, int32_t num_heads,
                                int32_t max_seq_len, float softmax_scale, void *out, float *lse,
                                void *workspace, size_t workspace_bytes, int32_t *dev_status,
                                void *stream);
mla_status_t mla_combine_planned(void *workspace, size_t workspace_bytes, int32_t batch,
                                 int32_t num_heads, void *out, float *lse, void *stream);

/*
 * mla_decode_append_planned — one decode step with its cache append fused in:
 * stores kv_new[b] (bf16 [batch, 576], the new latent row of request b) at
 * position seq_lens[b] - 1 of request b, i.e. at cache row
 * block_table[b][(L-1)/BS] * BS + (L-1) % BS, then decodes over the full
 * context, all in the decode kernel (requests with seq_lens[b] == 0 store
 * nothing).  Same result as mla_cache_append with that slot mapping followed
 * by mla_decode_planned; the cache must be writable.  A block-table entry
 * outside the pool is reported as MLA_ERR_DEVICE_RANGE and its row is not
 * stored.  For other slot mappings use mla_cache_append.
 */
mla_status_t mla_decode_append_planned(const void *q, void *cache, const void *kv_new,
                                       int64_t num_blocks, int32_t block_size,
                                       const int32_t *block_table, int32_t max_blocks_per_seq,
                                       const int32_t *seq_lens, int32_t batch, int32_t num_heads,
                                       int32_t max_seq_len, float softmax_scale, void *out,
                                       float *lse, void *workspace, size_t workspace_bytes,
                                       int32_t *dev_status, void *stream);

/*
 * mla_combine — merge split-KV partial results (flash-decoding).
 *
 * Partial w (one token range of one request) holds o_partial[w] = its own
 * normalised output and lse_partial[w] = log-sum-exp of its scores.  Request
 * b owns partials [split_offsets[b], split_offsets[b+1]) and gets
 *   M = max_w lse_w,  a_w = exp(lse_w - M),
 *   out[b,h,:] = sum_w a_w o_w[h,:] / sum_w a_w,   lse[b,h] = M + log sum_w a_w.
 * A partial with lse = -inf (an empty range) has no weight; a request with no
 * weighted partial gets out = 0, lse = -inf.  This regrouping of one softmax
 * over disjoint ranges is standard split-KV decoding, not on the pages; it is
 * how a long request is spread over many CTAs so it does not stall the batch
 * [dp-attention-expert-parallel-mla-kv-replication, "What it costs": a rank
 * holding long-context requests runs slower attention while others wait].
 *
 *   o_partial     fp32 [W, num_heads, 512];  lse_partial fp32 [W, num_heads]
 *   split_offsets int32 [batch + 1] (device), non-decreasing, last = W.
 *   out           bf16 [batch, num_heads, 512];  lse fp32 [batch, num_heads] or NULL.
 * Any num_heads >= 1.
 */
mla_status_t mla_combine(const float *o_partial, const float *lse_partial,
                         const int32_t *split_offsets, int32_t batch, int32_t num_heads,
                         void *out, float *lse, void *stream);

/*
 * FP8 latent cache — mla_cache_append_fp8, mla_decode_fp8, mla_decode_fp8_planned.
 *
 * Defined by: an FP8 MLA cache holds one byte per latent element, 576 bytes
 * per token per layer, half the bf16 cache [MLA 的 TP 切分 (10100.com),
 * opening paragraph (32 KB -> 576 bytes per token per layer) and section 5.1
 * ("576 bytes in FP8")].  The pages name no format, scale or rounding; this
 * library reads them as:
 *   - format: OCP FP8 E4M3 (bias 7, 3 mantissa bits, no infinities, code
 *     S.1111.111 is NaN, largest finite magnitude 448);
 *   - one scale per layer, kv_scale > 0 and finite (1 when unused): a stored
 *     code c stands for value(c) * kv_scale, so a row stays 576 bytes;
 *   - a new bf16 element x is stored as the code nearest to
 *     fp32(x) * fp32(1 / kv_scale) (one fp32 rounding each), ties to the even
 *     code, magnitudes above 448 saturating to 448, NaN to NaN.
 * Decode computes the same softmax attention as mla_decode (the equation at
 * the top of this file) over rows whose elements are value(code) * kv_scale.
 * The tensor cores run it on f16 operands, which hold every E4M3 value
 * exactly; q is taken to f16 inside the kernel, exactly for |q| in
 * [2^-14, 65504] (smaller magnitudes round to f16 subnormals, larger ones
 * saturate), so q must lie within 65504 in magnitude.
 *
 * mla_cache_append_fp8 — as mla_cache_append, storing each bf16 row of kv_new
 * (bf16 [num_tokens, 576]) quantised into cache8 (uint8 [num_blocks,
 * block_size, 576]) at its slot (-1 = skip; out-of-pool slots are skipped and
 * reported as MLA_ERR_DEVICE_RANGE in *dev_status).
 *
 * mla_decode_fp8 — mla_decode over cache8: plans (as mla_decode_plan, with the
 * table), decodes and merges split partials.  num_heads must be 128.
 *
 * mla_decode_fp8_planned — the same with the plan already in the workspace
 * (mla_decode_plan with the same lengths, table and sizes).  With kv_new
 * non-null (bf16 [batch, 576]) it first stores kv_new[b], quantised as above,
 * at position seq_lens[b] - 1 of request b inside the decode kernel, as
 * mla_decode_append_planned does for a bf16 cache.
 *
 * Arguments not listed are those of mla_decode / mla_decode_planned, with the
 * same layout, ownership and requirements (cache8 16-byte aligned; block_size
 * in {16, 32, 64, 128, 256}).  Returns MLA_OK, MLA_ERR_INVALID_ARGUMENT
 * (including a kv_scale that is not positive and finite),
 * MLA_ERR_UNSUPPORTED (num_heads != 128), MLA_ERR_WORKSPACE_TOO_SMALL or
 * MLA_ERR_CUDA; device faults go to *dev_status as for mla_decode.
 */
mla_status_t mla_cache_append_fp8(const void *kv_new, const int64_t *slot_mapping,
                                  int64_t num_tokens, void *cache8, int64_t num_blocks,
                                  int32_t block_size, float kv_scale, int32_t *dev_status,
                                  void *stream);
mla_status_t mla_decode_fp8(const void *q, const void *cache8, int64_t num_blocks,
                            int32_t block_size, const int32_t *block_table,
                            int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t batch,
                            int32_t num_heads, int32_t max_seq_len, float softmax_scale,
                            float kv_scale, void *out, float *lse, void *workspace,
                            size_t workspace_bytes, int32_t *dev_status, void *stream);
mla_status_t mla_decode_fp8_planned(const void *q, void *cache8, const void *kv_new,
                                    int64_t num_blocks, int32_t block_size,
                                    const int32_t *block_table, int32_t max_blocks_per_seq,
                                    const int32_t *seq_lens, int32_t batch, int32_t num_heads,
                                    int32_t max_seq_len, float softmax_scale, float kv_scale,
                                    void *out, float *lse, void *workspace, size_t workspace_bytes,
                                    int32_t *dev_status, void *stream);

/*
 * mla_decode_noalloc — mla_decode for callers that cannot allocate device
 * memory.  The pages have no counterpart to this entry point; it exists for
 * users of this library.
 *
 * Some callers cannot call cudaMalloc (or any allocating routine) at decode
 * time: code running inside a host framework that owns all device memory and
 * hands a plugin only its inputs and outputs, or a latency-critical serving
 * path that must not touch the allocator (and so cannot fail with
 * out-of-memory) in the middle of a step.  Such a caller cannot provide the
 * workspace mla_decode needs.  This entry point takes the same arguments as
 * mla_decode minus the workspace, and uses instead a fixed scratch array of
 * MLA_NOALLOC_SCRATCH_BYTES (16 MiB) compiled into the library as a
 * file-scope device array: every GPU that loads the library holds those
 * 16 MiB until the process exits.  It calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *
 * Limits: num_heads must be 128 (other values return MLA_ERR_UNSUPPORTED;
 * mla_decode takes 1 to 128); batch <=
 * MLA_NOALLOC_MAX_BATCH (8192), else MLA_ERR_INVALID_ARGUMENT with an
 * explanatory detail.  Because the scratch holds fewer split partials than a
 * full workspace, long contexts are spread over fewer SMs than with
 * mla_decode, which can make it slower; results agree with mla_decode within
 * the library's tolerance (the split points differ, so fp32 rounding
 * differs).
 *
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current.  Under CUDA's lazy module
 * loading that lookup may be the moment the driver loads the library's
 * device code and places the 16 MiB array on the device, so the first call
 * can itself fail with MLA_ERR_CUDA (out of memory).  Make one call per
 * device at set-up time (any valid call, e.g. batch 1), before any stream
 * capture and before the serving loop.  The address is kept per device and
 * looked up again only if the device's context was destroyed and recreated
 * (cudaDeviceReset); such a call again counts as a first call.
 *
 * Sharing: every call shares the one array and overwrites what the previous
 * call left there (each call re-plans and re-zeroes what must start at
 * zero), so calls whose kernels overlap on the GPU — on different streams, or
 * from different host threads — race and give undefined results: serialise
 * them.
 */
#define MLA_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
#define MLA_NOALLOC_MAX_BATCH 8192
mla_status_t mla_decode_noalloc(const void *q, const void *cache, int64_t num_blocks,
                                int32_t block_size, const int32_t *block_table,
                                int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                int32_t batch, int32_t num_heads, int32_t max_seq_len,
                                float softmax_scale, void *out, float *lse, int32_t *dev_status,
                                void *stream);

/*
 * mla_absorb_q / mla_absorb_out — the absorption GEMMs on either side of the
 * absorbed-form decode.  In decode each head's query is projected into the
 * latent space and the head attends over the shared latent directly
 * [dp-attention-expert-parallel-mla-kv-replication (inferenceinterviews.com),
 * "A strong answer"]; the head's 128 non-rotary query dims and its 128 value
 * dims map to the 512-dim latent through W_UK and W_UV, and the 64 rotary
 * dims are shared [MLA 的 TP 切分 (10100.com), §2.2].
 *
 * mla_absorb_q:   q[b,h,0:512]   = q_nope[b,h,:] . W_UK[h]   (fp32 sums)
 *                 q[b,h,512:576] = q_pe[b,h,:]                (copied)
 *   q_nope  device bf16 [B, 128, 128]   w_uk device bf16 [128, 128, 512]
 *   q_pe    device bf16 [B, 128, 64]    q    device bf16 [B, 128, 576], written
 * mla_absorb_out: o[b,h,:] = out[b,h,:] . W_UV[h]             (fp32 sums)
 *   out     device bf16 [B, 128, 512]   w_uv device bf16 [128, 512, 128]
 *   o       device bf16 [B, 128, 128], written
 *
 * All row-major and contiguous, 16-byte aligned; num_heads must be 128; any
 * B >= 0.  Each is one launch of a tensor-core kernel on `stream` (one CTA
 * per head and column tile streams the head's weight through TMA); nothing is
 * allocated and nothing is synchronised, so the calls can be captured.  The
 * launch is a programmatic dependent of the previous kernel on the stream: it
 * may start streaming the weight (which must not be written by that kernel)
 * before that kernel ends; it reads the activations and writes its output
 * only once that kernel has completed.
 *
 * dev_status (device int32, nullable) receives MLA_ERR_DEVICE_TIMEOUT (first
 * error wins) if one of the kernel's bounded waits runs out (100 ms each); the
 * block then stores nothing, waits (bounded) for its issued copies and MMAs
 * and returns, and the output is undefined.
 *
 * Returns MLA_OK (B = 0: nothing enqueued), MLA_ERR_INVALID_ARGUMENT
 * (B < 0, null or misaligned pointers), MLA_ERR_UNSUPPORTED (num_heads), or
 * MLA_ERR_CUDA.
 */
mla_status_t mla_absorb_q(const void *q_nope, const void *q_pe, const void *w_uk, int32_t batch,
                          int32_t num_heads, void *q, int32_t *dev_status, void *stream);
mla_status_t mla_absorb_out(const void *out, const void *w_uv, int32_t batch, int32_t num_heads,
                            void *o, int32_t *dev_status, void *stream);

/*
 * mla_place_requests — KV-load-aware placement of requests on data-parallel
 * attention ranks (host only; no GPU, no CUDA call).
 *
 * Under DP attention every rank decodes its own requests, and the MoE
 * all-to-all that follows attention keeps the ranks in lockstep, so a step
 * lasts as long as the rank with the most cache to read.  A rank holding the
 * long-context requests slows every rank, and long requests have to be
 * spread over the ranks [dp-attention-expert-parallel-mla-kv-replication
 * (inferenceinterviews.com), "What it costs" and "What interviewers probe
 * next"].  A decode reads every cached latent row of a request, so a rank's
 * load is the sum of its requests' cached tokens.
 *
 * Requests are placed longest first (ties: lower index first), each on the
 * rank with the least load so far (ties: lower rank), provided that rank's
 * load plus the request stays within capacity_tokens (0: no limit).  When
 * the least loaded rank cannot take it, no rank can, and the request is left
 * unplaced (rank_of = -1).  This is list scheduling in decreasing order
 * (Graham 1969): with no capacity limit the largest load is at most
 * (4/3 - 1/(3 ranks)) times the smallest achievable.
 *
 *   kv_tokens   host int64 [n]: cached tokens of request i (>= 0)
 *   n           number of requests (>= 0; 0 places nothing)
 *   ranks       number of DP ranks (>= 1)
 *   capacity_tokens  per-rank limit on the load (>= 0; 0: none)
 *   rank_of     host int32 [n], written: the rank of request i, or -1
 *   rank_load   host int64 [ranks], written: each rank's load
 *   unplaced    host int32, nullable: written with the number of -1 entries
 *
 * Returns MLA_OK, or MLA_ERR_INVALID_ARGUMENT (n < 0, ranks < 1, a negative
 * length or capacity, or a null array that is needed) with nothing written.
 * The caller owns every array; the library keeps nothing.
 */
mla_status_t mla_place_requests(const int64_t *kv_tokens, int32_t n, int32_t ranks,
                                int64_t capacity_tokens, int32_t *rank_of, int64_t *rank_load,
                                int32_t *unplaced);

/*
 * mla_place_one — the online form: the rank a new request of kv_tokens cached
 * tokens goes to, given the ranks' current loads (the least loaded, ties:
 * lower rank), or -1 in *rank when that rank's load plus the request exceeds
 * capacity_tokens (0: no limit).  rank_load is not changed.
 *
 * Returns MLA_OK, or MLA_ERR_INVALID_ARGUMENT (ranks < 1, a null pointer, a
 * negative length, load or capacity).
 */
mla_status_t mla_place_one(const int64_t *rank_load, int32_t ranks, int64_t capacity_tokens,
                           int64_t kv_tokens, int32_t *rank);

/*
 * mla_selftest_wait_timeout — checks, on the device, the bounded waits every
 * kernel of this library uses, without a fault or a hang.  One block of two
 * warps: warp 0 waits on an mbarrier that nothing arrives at, with a budget
 * of budget_ns; when it gives up it raises the block's abort flag and
 * reports MLA_ERR_DEVICE_TIMEOUT into *dev_status (first error wins).  Warp 1
 * waits on another such barrier through the decode kernel's own wait (100 ms
 * budget, ended early by the abort flag).  elapsed_ns[0..1] (device, uint64)
 * receive each warp's wait time in ns (0 if its wait completed).  The kernel
 * returns normally; the context stays usable.  Asynchronous on `stream`.
 *
 * Returns MLA_OK, MLA_ERR_INVALID_ARGUMENT (budget_ns outside 1 us .. 1 s,
 * a null or misaligned pointer) or MLA_ERR_CUDA (launch failure).
 */
mla_status_t mla_selftest_wait_timeout(uint64_t budget_ns, int32_t *dev_status,
                                       uint64_t *elapsed_ns, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */
