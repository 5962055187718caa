// gate_up.cu -- the gated-MLP activation Y = silu(G) * U on a GEMM output.
//
// For the MLP input projection the quantised weight is [2F, K] (gate rows
// [0, F), up rows [F, 2F)); nvfp4_linear_silu_mul computes G and U with the
// linear-layer path and applies silu(g) * u = g / (1 + e^-g) * u.  On the
// W4A4 branch (bf16 output, F % 128 == 0) the W4A4 kernel applies it in its
// epilogue; otherwise the GEMM writes fp32 [M, 2F] into the workspace and
// this kernel applies it.
#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;

// One row per blockIdx.y step, 4 features per thread; y2 is fp32 [M, 2F].
template <bool kF32>
__global__ void __launch_bounds__(kThreads)
silu_mul_kernel(const float* __restrict__ y2, int64_t M, int64_t F, void* __restrict__ y) {
  griddep_wait();  // y2 comes from the GEMM just before
  const int64_t f = ((int64_t)blockIdx.x * kThreads + threadIdx.x) * 4;
  if (f >= F) return;
  const bool vec = (F % 4 == 0) && f + 4 <= F;
  for (int64_t m = blockIdx.y; m < M; m += gridDim.y) {
    const float* g = y2 + m * 2 * F + f;
    const float* u = g + F;
    float o[4];
    if (vec) {
      const float4 gv = *reinterpret_cast<const float4*>(g), uv = *reinterpret_cast<const float4*>(u);
      o[0] = silu_mul(gv.x, uv.x);
      o[1] = silu_mul(gv.y, uv.y);
      o[2] = silu_mul(gv.z, uv.z);
      o[3] = silu_mul(gv.w, uv.w);
    } else {
      for (int e = 0; e < 4; ++e) o[e] = f + e < F ? silu_mul(g[e], u[e]) : 0.0f;
    }
    if (kF32) {
      float* out = static_cast<float*>(y) + m * F + f;
      if (vec) *reinterpret_cast<float4*>(out) = make_float4(o[0], o[1], o[2], o[3]);
      else
        for (int e = 0; e < 4 && f + e < F; ++e) out[e] = o[e];
    } else {
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(y) + m * F + f;
      if (vec) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(o[0], o[1]), hi = __floats2bfloat162_rn(o[2], o[3]);
        *reinterpret_cast<uint2*>(out) =
            make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
      } else {
        for (int e = 0; e < 4 && f + e < F; ++e) out[e] = __float2bfloat16_rn(o[e]);
      }
    }
  }
}

}  // namespace

cudaError_t launch_silu_mul(const float* y2, int64_t M, int64_t F, void* y, bool out_f32, cudaStream_t stream) {
  if (M <= 0 || F <= 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((F + 4 * kThreads - 1) / (4 * kThreads)), (unsigned)std::min<int64_t>(M, 65535));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (out_f32) return cudaLaunchKernelEx(&cfg, silu_mul_kernel<true>, y2, M, F, y);
  return cudaLaunchKernelEx(&cfg, silu_mul_kernel<false>, y2, M, F, y);
}

}  // namespace nvfp4
