// Backward of the LM head fused with the loss (vpce_lmhead_backward).
//
// The forward never wrote the logits, so the backward forms them again: per
// chunk of rows, the tensor-core kernel recomputes each logits tile and
// writes dZ = (softmax - onehot) * g as bf16 (the epilogue uses the
// forward's logsumexp and n_valid); then two plain GEMMs through cuBLAS give
//     dX[chunk]  = sum_i dZ_i W_i          (fp32, then rounded to bf16)
//     dW_i      += dZ_i^T X[chunk]         (fp32, accumulated)
// The chunk bounds the dZ scratch to rows x V bf16 (1.05 GB for the default
// 4096 rows at V = 128256; a smaller workspace gives smaller chunks, down to
// 128 rows), the "do not assemble the big tensor" of the CMU notes (§5.5)
// applied to the gradient.  Larger chunks give cuBLAS larger products.
#include <cublas_v2.h>

#include <mutex>

#include "vpce_kernels.cuh"

namespace vpce {

bool launch_gemm_grad(const void* x, long long ld_x, const void* const* w, long long ld_w, int t, long long s,
                      long long h, const long long* vocab_start, const long long* targets, long long ignore_index,
                      const float* lse, const float* grad_rows, float grad, unsigned short* dz, long long ldz,
                      Header* hdr, int sms, cudaStream_t st);

namespace {

constexpr long long kBwdRows = 4096;  // rows per chunk with the suggested workspace
constexpr long long kMinBwdRows = 128;
// cuBLAS's own scratch, carved from the caller's workspace so that no call
// allocates (and a stream capture records nothing but kernels).
constexpr size_t kBlasBytes = size_t(32) << 20;

__global__ void f32_to_bf16_rows(const float* src, long long lds, __nv_bfloat16* dst, long long ldd, long long rows,
                                 long long cols) {
  const long long n = rows * cols;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (long long)gridDim.x * blockDim.x) {
    const long long r = e / cols, c = e - r * cols;
    dst[r * ldd + c] = __float2bfloat16_rn(src[r * lds + c]);
  }
}

std::mutex g_blas_mu;
cublasHandle_t g_blas[64] = {};

cublasHandle_t blas_handle(int dev) {
  if (dev < 0 || dev >= 64) return nullptr;
  if (g_blas[dev] == nullptr) {
    cublasHandle_t hnd = nullptr;
    if (cublasCreate(&hnd) != CUBLAS_STATUS_SUCCESS) return nullptr;
    g_blas[dev] = hnd;
  }
  return g_blas[dev];
}

}  // namespace

long long lmhead_bwd_ldz(long long V) { return (V + 7) / 8 * 8; }

size_t lmhead_bwd_bytes_for(long long rows, long long V, long long h) {
  return round256(size_t(rows) * size_t(lmhead_bwd_ldz(V)) * 2u) + round256(size_t(rows) * size_t(h) * 4u) +
         kBlasBytes;
}

size_t lmhead_bwd_workspace_bytes(long long V, long long h) { return lmhead_bwd_bytes_for(kBwdRows, V, h); }
size_t lmhead_bwd_min_workspace_bytes(long long V, long long h) { return lmhead_bwd_bytes_for(kMinBwdRows, V, h); }

// The largest chunk (a multiple of kMinBwdRows, at most kBwdRows) whose
// scratch fits in `bytes`.
long long lmhead_bwd_rows_for(size_t bytes, long long V, long long h) {
  long long r = kBwdRows;
  while (r > kMinBwdRows && lmhead_bwd_bytes_for(r, V, h) > bytes) r -= kMinBwdRows;
  return r;
}

// Returns VPCE_OK, VPCE_ERR_CUDA (a launch or a cuBLAS call failed).
vpce_status lmhead_backward_run(const void* x, long long ld_x, const void* const* w, long long ld_w, int t,
                                long long s, long long h, const long long* vs, const long long* targets,
                                long long ignore_index, float grad, const float* grad_rows, const float* lse,
                                Header* hdr, void* dx, long long ld_dx, float* const* dw, long long ld_dw, void* ws,
                                size_t ws_bytes, int sms, cudaStream_t st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return VPCE_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_blas_mu);
  cublasHandle_t hb = blas_handle(dev);
  const long long V = vs[t];
  const long long ldz = lmhead_bwd_ldz(V);
  const long long rows = lmhead_bwd_rows_for(ws_bytes, V, h);
  unsigned short* dz = static_cast<unsigned short*>(ws);
  unsigned char* dx32_at = static_cast<unsigned char*>(ws) + round256(size_t(rows) * size_t(ldz) * 2u);
  float* dx32 = reinterpret_cast<float*>(dx32_at);
  void* blas_ws = dx32_at + round256(size_t(rows) * size_t(h) * 4u);
  // setting the stream resets cuBLAS to its default workspace pool, so the
  // caller's slice is installed after it, on every call
  if (hb == nullptr || cublasSetStream(hb, st) != CUBLAS_STATUS_SUCCESS ||
      cublasSetWorkspace(hb, blas_ws, kBlasBytes) != CUBLAS_STATUS_SUCCESS)
    return VPCE_ERR_CUDA;
  const float one = 1.f, zero = 0.f;
  for (long long r0 = 0; r0 < s; r0 += rows) {
    const long long R = s - r0 < rows ? s - r0 : rows;
    const unsigned char* xr = static_cast<const unsigned char*>(x) + r0 * ld_x * 2;
    if (!launch_gemm_grad(xr, ld_x, w, ld_w, t, R, h, vs, targets + r0, ignore_index, lse + r0,
                          grad_rows != nullptr ? grad_rows + r0 : nullptr, grad, dz, ldz, hdr, sms, st))
      return VPCE_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return VPCE_ERR_CUDA;
    for (int i = 0; i < t; ++i) {
      const int wi = int(vs[i + 1] - vs[i]);
      // column-major: dX^T [h, R] (+)= W_i^T [h, w_i] * dZ_i^T [w_i, R]
      if (cublasGemmEx(hb, CUBLAS_OP_N, CUBLAS_OP_N, int(h), int(R), wi, &one, w[i], CUDA_R_16BF, int(ld_w),
                       dz + vs[i], CUDA_R_16BF, int(ldz), i == 0 ? &zero : &one, dx32, CUDA_R_32F, int(h),
                       CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
        return VPCE_ERR_CUDA;
      // column-major: dW_i^T [h, w_i] += X^T [h, R] * dZ_i [R, w_i]
      if (cublasGemmEx(hb, CUBLAS_OP_N, CUBLAS_OP_T, int(h), wi, int(R), &one, xr, CUDA_R_16BF, int(ld_x),
                       dz + vs[i], CUDA_R_16BF, int(ldz), &one, dw[i], CUDA_R_32F, int(ld_dw), CUBLAS_COMPUTE_32F,
                       CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
        return VPCE_ERR_CUDA;
    }
    const long long n = R * h;
    long long blocks = (n + 255) / 256;
    if (blocks > (long long)sms * 16) blocks = (long long)sms * 16;
    f32_to_bf16_rows<<<int(blocks), 256, 0, st>>>(dx32, h,
                                                   static_cast<__nv_bfloat16*>(dx) + r0 * ld_dx, ld_dx, R, h);
    if (cudaGetLastError() != cudaSuccess) return VPCE_ERR_CUDA;
  }
  return VPCE_OK;
}

}  // namespace vpce
