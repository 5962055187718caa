// gemm_w4a16_any.cu -- W4A16 (bf16 activations x NVFP4 weights, fp32
// accumulation) for weights whose K is a multiple of 16 but not of 64.
//
// "SOAR 2026 Recap ...", section "1. Quantization and GEMM dispatch" (W4A16
// below the crossover); NVFP4 blocks are 16 elements, so any K % 16 == 0 is a
// valid weight.  The tensor-core kernels stream 64-wide chunks by TMA and need
// code rows that are multiples of 32 bytes; rows of 8 * odd bytes (K = 16 *
// odd) cannot be described to the TMA at all.  This kernel covers those
// shapes with plain loads: correctness first, for layers that are rare.
//
// One warp per (weight row n, group of up to 8 tokens).  Lane l takes the
// 16-element blocks b = l, l + 32, ...: value(code) * value(scale) exactly in
// binary32 (at most 2 + 4 significant bits), times x (bf16, exact in
// binary32), fma-accumulated per token in block order; then a shuffle tree
// over the lanes (offsets 16, 8, 4, 2, 1), times ts, rounded to the output
// type.  Programmatic dependent launch: the wait comes before any read.
#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTok = 8;  // tokens per warp

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <bool kF32>
__global__ void __launch_bounds__(kThreads)
w4a16_any_kernel(const uint4* __restrict__ x, const uint8_t* __restrict__ codes, const uint8_t* __restrict__ smma,
                 const float* __restrict__ ts_ptr, int64_t M, int64_t N, int64_t K, void* __restrict__ y) {
  griddep_wait();
  const float ts = *ts_ptr;
  const int lane = threadIdx.x & 31;
  const int64_t kb = K / 16, ct = (kb + 3) / 4, groups = (M + kTok - 1) / kTok;
  const int64_t xrow = K / 8;  // 16-byte pieces per token row
  for (int64_t w = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); w < N * groups;
       w += (int64_t)gridDim.x * kWarps) {
    const int64_t n = w / groups, m0 = (w - n * groups) * kTok;
    const int mt = (int)min((int64_t)kTok, M - m0);
    float acc[kTok];
#pragma unroll
    for (int t = 0; t < kTok; ++t) acc[t] = 0.0f;
    for (int64_t b = lane; b < kb; b += 32) {
      const uint2 cw = *reinterpret_cast<const uint2*>(codes + n * (K / 2) + 8 * b);
      const float s = e4m3_to_f32(smma[scale_mma_offset(n, b, ct)]);
      float wv[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t code = ((j < 8 ? cw.x : cw.y) >> (4 * (j & 7))) & 15u;
        const float mag = e2m1_mag_to_f32(code & 7u);
        wv[j] = __fmul_rn(code & 8u ? -mag : mag, s);
      }
#pragma unroll
      for (int t = 0; t < kTok; ++t) {
        if (t < mt) {
          const uint4* xp = x + (m0 + t) * xrow + 2 * b;
          const uint4 v0 = __ldg(xp), v1 = __ldg(xp + 1);
          const uint32_t xw[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
          float a = acc[t];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            a = __fmaf_rn(wv[2 * j], bf16_lo(xw[j]), a);
            a = __fmaf_rn(wv[2 * j + 1], bf16_hi(xw[j]), a);
          }
          acc[t] = a;
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kTok; ++t) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[t] = __fadd_rn(acc[t], __shfl_xor_sync(0xffffffffu, acc[t], off));
    }
    if (lane < mt) {
      float v = 0.0f;
#pragma unroll
      for (int t = 0; t < kTok; ++t)
        if (t == lane) v = acc[t];
      v = __fmul_rn(v, ts);
      const int64_t o = (m0 + lane) * N + n;
      if (kF32) static_cast<float*>(y)[o] = v;
      else static_cast<__nv_bfloat16*>(y)[o] = __float2bfloat16_rn(v);
    }
  }
}

}  // namespace

cudaError_t launch_gemm_w4a16_any(const void* x, int64_t M, const uint8_t* codes, const uint8_t* scales_mma,
                                  const float* ts, int64_t N, int64_t K, void* y, bool out_f32, int num_sms,
                                  cudaStream_t stream) {
  if (M <= 0) return cudaSuccess;
  if (K < 16 || K % 16 != 0) return cudaErrorNotSupported;
  const int64_t warps = N * ((M + kTok - 1) / kTok);
  const int64_t grid = std::min<int64_t>((warps + kWarps - 1) / kWarps, (int64_t)num_sms * 16);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::max<int64_t>(grid, 1));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  auto kern = out_f32 ? w4a16_any_kernel<true> : w4a16_any_kernel<false>;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<const uint4*>(x), codes, scales_mma, ts, M, N, K, y);
}

}  // namespace nvfp4
