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
// Both are plain batched GEMMs over the heads (per head [B x 128] x [128 x 512]
// and [B x 512] x [512 x 128], bf16 in, fp32 accumulation, bf16 out): they run
// on cuBLAS (strided batched, one call each), with one handle and one fixed
// workspace per device, made on the first call.
#include <cublas_v2.h>

#include <mutex>

#include "common.cuh"

namespace mla {
void set_error_detail(const char *msg);

namespace {

constexpr int kNope = 128;   // non-rotary query dims per head
constexpr int kRope = 64;    // shared rotary dims
constexpr int kVHead = 128;  // value dims per head after W_UV
constexpr size_t kCublasWorkspace = 32u << 20;

struct Blas {
  cublasHandle_t handle = nullptr;
  void *workspace = nullptr;
  std::mutex mu;  // a handle is used by one thread at a time
};

Blas g_blas[64];
std::mutex g_blas_mu;

// The device's handle (created with its workspace on first use; its stream is
// set per call), or nullptr.
Blas *blas_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(g_blas_mu);
  Blas &b = g_blas[dev];
  if (!b.handle) {
    cublasHandle_t h = nullptr;
    if (cublasCreate(&h) != CUBLAS_STATUS_SUCCESS) return nullptr;
    void *ws = nullptr;
    if (cudaMalloc(&ws, kCublasWorkspace) != cudaSuccess ||
        cublasSetWorkspace(h, ws, kCublasWorkspace) != CUBLAS_STATUS_SUCCESS) {
      if (ws) cudaFree(ws);
      cublasDestroy(h);
      return nullptr;
    }
    b.handle = h;
    b.workspace = ws;
  }
  return &b;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// Row-major C[h] = A[h] (B x K) . W[h] (K x N) for every head h, written as the
// column-major product C^T = W^T A^T that cuBLAS computes: W[h] row-major is W^T
// column-major with leading dimension N, A and C rows are `lda` / `ldc` apart.
mla_status_t batched(const void *a, int64_t lda, int64_t stride_a, const void *w, int n, int k,
                     void *c, int64_t ldc, int64_t stride_c, int batch, int heads, void *stream,
                     const char *what) {
  Blas *b = blas_for_current_device();
  if (!b) {
    set_error_detail("cuBLAS handle creation failed");
    return MLA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(b->mu);
  const float one = 1.f, zero = 0.f;
  cublasStatus_t s = cublasSetStream(b->handle, (cudaStream_t)stream);
  if (s == CUBLAS_STATUS_SUCCESS)
    s = cublasGemmStridedBatchedEx(b->handle, CUBLAS_OP_N, CUBLAS_OP_N, n, batch, k, &one, w,
                                   CUDA_R_16BF, n, (int64_t)k * n, a, CUDA_R_16BF, (int)lda,
                                   stride_a, &zero, c, CUDA_R_16BF, (int)ldc, stride_c, heads,
                                   CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
  if (s != CUBLAS_STATUS_SUCCESS) {
    set_error_detail(what);
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" {

mla_status_t mla_absorb_q(const void *q_nope, const void *q_pe, const void *w_uk, int32_t batch,
                          int32_t num_heads, void *q, void *stream) {
  set_error_detail("");
  if (batch < 0 || num_heads != kHeads) {
    set_error_detail("batch < 0 or num_heads != 128");
    return batch < 0 ? MLA_ERR_INVALID_ARGUMENT : MLA_ERR_UNSUPPORTED;
  }
  if (batch == 0) return MLA_OK;
  if (!q_nope || !q_pe || !w_uk || !q) {
    set_error_detail("null pointer");
    return MLA_ERR_INVALID_ARGUMENT;
  }
  if (!aligned16(q_nope) || !aligned16(q_pe) || !aligned16(w_uk) || !aligned16(q)) {
    set_error_detail("pointers must be 16-byte aligned");
    return MLA_ERR_INVALID_ARGUMENT;
  }
  // q[b, h, 0:512] = q_nope[b, h, :] . W_UK[h]
  mla_status_t s = batched(q_nope, (int64_t)kHeads * kNope, kNope, w_uk, kVDim, kNope, q,
                           (int64_t)kHeads * kRow, kRow, batch, kHeads, stream,
                           "cuBLAS batched GEMM (q_nope . W_UK) failed");
  if (s != MLA_OK) return s;
  // q[b, h, 512:576] = q_pe[b, h, :]
  const cudaError_t e = cudaMemcpy2DAsync(
      static_cast<__nv_bfloat16 *>(q) + kVDim, kRow * sizeof(__nv_bfloat16), q_pe,
      kRope * sizeof(__nv_bfloat16), kRope * sizeof(__nv_bfloat16), (size_t)batch * kHeads,
      cudaMemcpyDeviceToDevice, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    set_error_detail(cudaGetErrorString(e));
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

mla_status_t mla_absorb_out(const void *out, const void *w_uv, int32_t batch, int32_t num_heads,
                            void *o, void *stream) {
  set_error_detail("");
  if (batch < 0 || num_heads != kHeads) {
    set_error_detail("batch < 0 or num_heads != 128");
    return batch < 0 ? MLA_ERR_INVALID_ARGUMENT : MLA_ERR_UNSUPPORTED;
  }
  if (batch == 0) return MLA_OK;
  if (!out || !w_uv || !o) {
    set_error_detail("null pointer");
    return MLA_ERR_INVALID_ARGUMENT;
  }
  if (!aligned16(out) || !aligned16(w_uv) || !aligned16(o)) {
    set_error_detail("pointers must be 16-byte aligned");
    return MLA_ERR_INVALID_ARGUMENT;
  }
  // o[b, h, :] = out[b, h, :] . W_UV[h]
  return batched(out, (int64_t)kHeads * kVDim, kVDim, w_uv, kVHead, kVDim, o,
                 (int64_t)kHeads * kVHead, kVHead, batch, kHeads, stream,
                 "cuBLAS batched GEMM (out . W_UV) failed");
}

}  // extern "C"
