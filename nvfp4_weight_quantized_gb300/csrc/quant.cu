// quant.cu -- NVFP4 quantisers: FourOverSix for weights, M=6 for activations.
//
// Method: "SOAR Weekly Champion Notes 07 ... NVFP4 Quantization Improvements",
// section "02 FourOverSix" -- per block, the M=4 scale is the FP8 rounding of
// the M=6 scale times 1.5; both candidates are dequantised and the one with
// the smaller block MSE is kept (M=4 only when strictly smaller).  Section
// "01 Background" gives the E2M1 grid and the M=6 normalisation to [-6, 6].
//
// Two launches per tensor:
//   1. amax_partial_kernel: a grid-stride max of |x| over the tensor, one
//      partial per CTA in the workspace (bf16 magnitude bits: the unsigned
//      order of those bits is the order of the values, and Inf/NaN sort
//      above every finite value, which is how non-finite input is detected).
//   2. quant_kernel<FOS>: every CTA folds the partials into the tensor scale
//      ts = amax / divisor, then each thread quantises whole 16-element
//      blocks (32 bytes of bf16 in, 8 bytes of codes + 1 scale out), fully
//      coalesced 128-bit loads.
// Every binary32 step uses the explicit round-to-nearest intrinsics, so the
// compiler cannot contract multiply-adds and the result is bit-identical to
// the order of operations stated in nvfp4.h.
#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t block_reduce_max(uint32_t v, uint32_t* red) {
  v = __reduce_max_sync(0xffffffffu, v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < (int)(blockDim.x >> 5) ? red[lane] : 0u;
    w = __reduce_max_sync(0xffffffffu, w);
    if (lane == 0) red[0] = w;
  }
  __syncthreads();
  return red[0];
}

__global__ void __launch_bounds__(kThreads)
amax_partial_kernel(const uint4* __restrict__ x, int64_t n_vec, uint32_t* __restrict__ partial,
                    unsigned long long* __restrict__ counter_to_clear) {
  __shared__ uint32_t red[kThreads / 32];
  uint32_t m2 = 0;  // two running maxima of bf16 magnitude bits, one per half
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n_vec; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = ld_stream_u4(x + i + u * stride);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      m2 = __vmaxu2(m2, v[u].x & 0x7FFF7FFFu);
      m2 = __vmaxu2(m2, v[u].y & 0x7FFF7FFFu);
      m2 = __vmaxu2(m2, v[u].z & 0x7FFF7FFFu);
      m2 = __vmaxu2(m2, v[u].w & 0x7FFF7FFFu);
    }
  }
  for (; i < n_vec; i += stride) {
    uint4 v = ld_stream_u4(x + i);
    m2 = __vmaxu2(m2, v.x & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, v.y & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, v.z & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, v.w & 0x7FFF7FFFu);
  }
  uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
  m = block_reduce_max(m, red);
  if (threadIdx.x == 0) {
    partial[blockIdx.x] = m;
    if (counter_to_clear != nullptr && blockIdx.x == 0) *counter_to_clear = 0ull;
  }
}

// Quantise one 16-element block with scale value `sv` (binary32 value of the
// E4M3 byte) and tensor scale ts.  ax[] holds |x|.  Returns the block SSE in
// the fixed tree order; mags[] receive the E2M1 magnitude codes.
__device__ __forceinline__ float block_sse(const float (&ax)[16], float sv, float ts,
                                           uint32_t (&mags)[16]) {
  const float eff = __fmul_rn(sv, ts);
  float e[16];
  if (eff == 0.0f) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      mags[i] = 0u;
      e[i] = __fmul_rn(ax[i], ax[i]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      float r0 = fminf(__fdiv_rn(ax[i], eff), 6.0f);
      float r1 = fminf(__fdiv_rn(ax[i + 1], eff), 6.0f);
      uint32_t p = cvt_e2m1x2(r1, r0);
      mags[i] = p & 7u;
      mags[i + 1] = (p >> 4) & 7u;
      float d0 = __fsub_rn(ax[i], __fmul_rn(e2m1_mag_to_f32(mags[i]), eff));
      float d1 = __fsub_rn(ax[i + 1], __fmul_rn(e2m1_mag_to_f32(mags[i + 1]), eff));
      e[i] = __fmul_rn(d0, d0);
      e[i + 1] = __fmul_rn(d1, d1);
    }
  }
  float a[8], b[4];
#pragma unroll
  for (int j = 0; j < 8; ++j) a[j] = __fadd_rn(e[j], e[j + 8]);
#pragma unroll
  for (int j = 0; j < 4; ++j) b[j] = __fadd_rn(a[j], a[j + 4]);
  return __fadd_rn(__fadd_rn(b[0], b[2]), __fadd_rn(b[1], b[3]));
}

template <bool kFos>
__global__ void __launch_bounds__(kThreads)
quant_kernel(const uint4* __restrict__ x, int64_t rows, int64_t K, const uint32_t* __restrict__ partial,
             int n_partial, float divisor, uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
             uint8_t* __restrict__ scales_mma, float* __restrict__ ts_out, uint8_t* __restrict__ choice,
             unsigned long long* __restrict__ m4_count, unsigned int* __restrict__ status) {
  __shared__ uint32_t red[kThreads / 32];
  uint32_t am = 0;
  for (int i = threadIdx.x; i < n_partial; i += blockDim.x) am = max(am, partial[i]);
  am = block_reduce_max(am, red);
  if (am >= 0x7F80u) {  // Inf or NaN somewhere in the tensor
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(status, kStatusNonfinite);
    return;
  }
  const float amax = __uint_as_float(am << 16);
  const float ts = amax == 0.0f ? 1.0f : __fdiv_rn(amax, divisor);
  if (blockIdx.x == 0 && threadIdx.x == 0) *ts_out = ts;

  const int64_t kb = K >> 4;
  const int64_t ct = (kb + 3) >> 2;
  const int64_t nblk = rows * kb;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  uint32_t n_m4 = 0;
  for (int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; blk < nblk; blk += stride) {
    const uint4 v0 = ld_stream_u4(x + 2 * blk);
    const uint4 v1 = ld_stream_u4(x + 2 * blk + 1);
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float ax[16];
    uint32_t sign = 0;  // bit i = sign of element i
    float bmax = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      ax[2 * j] = __uint_as_float((w[j] & 0x7FFFu) << 16);
      ax[2 * j + 1] = __uint_as_float(w[j] & 0x7FFF0000u);
      sign |= ((w[j] >> 15) & 1u) << (2 * j);
      sign |= ((w[j] >> 31) & 1u) << (2 * j + 1);
      bmax = fmaxf(bmax, fmaxf(ax[2 * j], ax[2 * j + 1]));
    }
    // s6 = E4M3((amax_block / 6) / ts)
    const float r6 = __fdiv_rn(__fdiv_rn(bmax, 6.0f), ts);
    const uint32_t s6 = cvt_e4m3x2(0.0f, r6) & 0xFFu;
    uint32_t mags[16];
    uint32_t s = s6;
    if (kFos) {
      const float s6v = e4m3_to_f32(s6);
      const uint32_t s4 = cvt_e4m3x2(0.0f, __fmul_rn(s6v, 1.5f)) & 0xFFu;
      uint32_t mags4[16];
      const float sse6 = block_sse(ax, s6v, ts, mags);
      const float sse4 = block_sse(ax, e4m3_to_f32(s4), ts, mags4);
      const bool m4 = sse4 < sse6;
      if (m4) {
#pragma unroll
        for (int i = 0; i < 16; ++i) mags[i] = mags4[i];
        s = s4;
        ++n_m4;
      }
      if (choice != nullptr) choice[blk] = m4 ? 1 : 0;
    } else {
      (void)block_sse(ax, e4m3_to_f32(s6), ts, mags);
    }
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) lo |= (mags[i] | (((sign >> i) & 1u) << 3)) << (4 * i);
#pragma unroll
    for (int i = 0; i < 8; ++i) hi |= (mags[8 + i] | (((sign >> (8 + i)) & 1u) << 3)) << (4 * i);
    *reinterpret_cast<uint2*>(codes + 8 * blk) = make_uint2(lo, hi);
    if (scales != nullptr) scales[blk] = (uint8_t)s;
    if (scales_mma != nullptr) {
      const int64_t r = blk / kb, c = blk - r * kb;
      scales_mma[scale_mma_offset(r, c, ct)] = (uint8_t)s;
    }
  }
  // zero the padding of the MMA scale tiling (rows up to a multiple of 128,
  // scale columns up to a multiple of 4)
  if (scales_mma != nullptr) {
    const int64_t rows_p = (rows + 127) & ~int64_t(127), cols_p = ct * 4;
    const int64_t pad_cols = cols_p - kb;
    const int64_t n_pad_a = rows * pad_cols;              // real rows, padded columns
    const int64_t n_pad_b = (rows_p - rows) * cols_p;     // padded rows, all columns
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_pad_a + n_pad_b; i += stride) {
      int64_t r, c;
      if (i < n_pad_a) {
        r = i / pad_cols;
        c = kb + (i - r * pad_cols);
      } else {
        const int64_t j = i - n_pad_a;
        r = rows + j / cols_p;
        c = j % cols_p;
      }
      scales_mma[scale_mma_offset(r, c, ct)] = 0;
    }
  }
  if (kFos && m4_count != nullptr) {
    n_m4 = __reduce_add_sync(0xffffffffu, n_m4);
    if ((threadIdx.x & 31) == 0 && n_m4) atomicAdd(m4_count, (unsigned long long)n_m4);
  }
}

}  // namespace

size_t quant_workspace_bytes() { return kMaxAmaxPartials * sizeof(uint32_t); }

cudaError_t launch_quantize(const void* x, int64_t rows, int64_t K, float divisor, bool fos,
                            uint8_t* codes, uint8_t* scales, uint8_t* scales_mma, float* ts,
                            uint8_t* choice, unsigned long long* m4_count, void* workspace,
                            unsigned int* status, int num_sms, cudaStream_t stream) {
  const int64_t n_vec = rows * K / 8;  // 16-byte vectors of bf16
  int g1 = (int)std::min<int64_t>((n_vec + kThreads * 4 - 1) / (kThreads * 4), (int64_t)num_sms * 4);
  g1 = std::max(1, std::min(g1, kMaxAmaxPartials));
  uint32_t* partial = static_cast<uint32_t*>(workspace);
  amax_partial_kernel<<<g1, kThreads, 0, stream>>>(static_cast<const uint4*>(x), n_vec, partial,
                                                   fos ? m4_count : nullptr);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int64_t nblk = rows * (K / 16);
  int g2 = (int)std::min<int64_t>((nblk + kThreads - 1) / kThreads, (int64_t)num_sms * 8);
  g2 = std::max(g2, 1);
  if (fos)
    quant_kernel<true><<<g2, kThreads, 0, stream>>>(static_cast<const uint4*>(x), rows, K, partial, g1,
                                                    divisor, codes, scales, scales_mma, ts, choice,
                                                    m4_count, status);
  else
    quant_kernel<false><<<g2, kThreads, 0, stream>>>(static_cast<const uint4*>(x), rows, K, partial, g1,
                                                     divisor, codes, scales, scales_mma, ts, nullptr,
                                                     nullptr, status);
  return cudaGetLastError();
}

}  // namespace nvfp4
