// qat.cu -- the backward pass of an NVFP4-forward linear layer (quantisation-
// aware training with the straight-through estimator).
//
// "SOAR 2026 Recap ...", section "3. EAGLE-3 speculative decoding and hybrid
// architecture adaptation", paragraph "NVFP4 QAT": the forward GEMM runs in
// FP4 itself (nvfp4_gemm_w4a4 here) and the backward pass sends the
// gradients straight through the quantisers to the bf16 master weights.  For
// Y = X_hat W_hat^T that gives dX = dY W_hat and dW = dY^T X_hat, plain bf16
// GEMMs: the NVFP4 operands are dequantised to bf16 by dequant_bf16_kernel
// and the two products run on cuBLAS (fp32 accumulation).
#include <cublas_v2.h>

#include <map>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;

// One 16-element block per thread and step: value(code) * value(scale) is
// exact in binary32 (at most 2 + 4 significant bits), times the tensor scale
// rounded once, then rounded to bf16; 8 code bytes in, 32 bytes out.
__global__ void __launch_bounds__(kThreads)
dequant_bf16_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ smma,
                    const float* __restrict__ ts_ptr, int64_t R, int64_t K, __nv_bfloat16* __restrict__ out) {
  griddep_wait();
  const float ts = *ts_ptr;
  const int64_t kb = K / 16, ct = (kb + 3) / 4, nblk = R * kb;
  for (int64_t b = (int64_t)blockIdx.x * kThreads + threadIdx.x; b < nblk; b += (int64_t)gridDim.x * kThreads) {
    const int64_t r = b / kb, c = b - r * kb;
    const uint2 cw = *reinterpret_cast<const uint2*>(codes + r * (K / 2) + 8 * c);
    const float s = e4m3_to_f32(smma[scale_mma_offset(r, c, ct)]);
    uint32_t o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t byte = ((j < 4 ? cw.x : cw.y) >> (8 * (j & 3))) & 0xFFu;
      float q[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t code = (byte >> (4 * h)) & 15u;
        const float mag = e2m1_mag_to_f32(code & 7u);
        q[h] = __fmul_rn(__fmul_rn(code & 8u ? -mag : mag, s), ts);
      }
      __nv_bfloat162 p = __floats2bfloat162_rn(q[0], q[1]);
      o[j] = *reinterpret_cast<uint32_t*>(&p);
    }
    uint4* dst = reinterpret_cast<uint4*>(out + r * K + 16 * c);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

std::mutex g_blas_mu;
std::map<int, cublasHandle_t> g_blas;  // per device, created on first use

cublasStatus_t blas_handle(cublasHandle_t* h) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CUBLAS_STATUS_NOT_INITIALIZED;
  auto it = g_blas.find(dev);
  if (it != g_blas.end()) {
    *h = it->second;
    return CUBLAS_STATUS_SUCCESS;
  }
  cublasStatus_t st = cublasCreate(h);
  if (st == CUBLAS_STATUS_SUCCESS) g_blas[dev] = *h;
  return st;
}

}  // namespace

cudaError_t launch_dequant_bf16(const uint8_t* codes, const uint8_t* scales_mma, const float* ts, int64_t R,
                                int64_t K, void* out, int num_sms, cudaStream_t stream) {
  if (R <= 0) return cudaSuccess;
  const int64_t nblk = R * (K / 16);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::min<int64_t>((nblk + kThreads - 1) / kThreads, (int64_t)num_sms * 8));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, dequant_bf16_kernel, codes, scales_mma, ts, R, K,
                            static_cast<__nv_bfloat16*>(out));
}

// Row-major operands seen by column-major cuBLAS: a row-major [r, c] matrix is
// a column-major [c, r] one with leading dimension c.
//   dX [M, K] = dY [M, N] W_hat [N, K]:  dX^T = W_hat^T dY^T  -> C[K, M] = A[K, N] B[N, M]
//   dW [N, K] = dY^T [N, M] X_hat [M, K]: dW^T = X_hat^T dY   -> C[K, N] = A[K, M] B^T, B = dY^T as [N, M]
int qat_backward_gemms(const void* dy, const void* w_hat, const void* x_hat, int64_t M, int64_t N, int64_t K,
                       void* dx, void* dw, cudaStream_t stream) {
  std::lock_guard<std::mutex> lk(g_blas_mu);
  cublasHandle_t h = nullptr;
  cublasStatus_t st = blas_handle(&h);
  if (st != CUBLAS_STATUS_SUCCESS) return (int)st;
  if ((st = cublasSetStream(h, stream)) != CUBLAS_STATUS_SUCCESS) return (int)st;
  const float one = 1.0f, zero = 0.0f;
  if (dx != nullptr) {
    st = cublasGemmEx(h, CUBLAS_OP_N, CUBLAS_OP_N, (int)K, (int)M, (int)N, &one, w_hat, CUDA_R_16BF, (int)K, dy,
                      CUDA_R_16BF, (int)N, &zero, dx, CUDA_R_16BF, (int)K, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
    if (st != CUBLAS_STATUS_SUCCESS) return (int)st;
  }
  if (dw != nullptr) {
    st = cublasGemmEx(h, CUBLAS_OP_N, CUBLAS_OP_T, (int)K, (int)N, (int)M, &one, x_hat, CUDA_R_16BF, (int)K, dy,
                      CUDA_R_16BF, (int)N, &zero, dw, CUDA_R_32F, (int)K, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
    if (st != CUBLAS_STATUS_SUCCESS) return (int)st;
  }
  return 0;
}

}  // namespace nvfp4
