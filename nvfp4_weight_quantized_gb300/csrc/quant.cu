// quant.cu -- NVFP4 quantisers: FourOverSix for weights, M=6 for activations.
//
// Method: "SOAR Weekly Champion Notes 07 ... NVFP4 Quantization Improvements",
// section "02 FourOverSix" -- per block, the M=4 scale is the FP8 rounding of
// the M=6 scale times 1.5; both candidates are dequantised and the one with
// the smaller block MSE is kept (M=4 only when strictly smaller).  Section
// "01 Background" gives the E2M1 grid and the M=6 normalisation to [-6, 6].
//
// Two launches per tensor by default (below); optionally one cooperative
// launch (quant_fused_kernel: read once, a grid-wide barrier for the tensor
// scale, quantise from shared memory; nvfp4_set_single_launch_quantizer):
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
#include <cooperative_groups.h>

#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;

// L2 policies: the amax pass marks the tensor "evict last" so that the
// quantisation pass that follows finds it in L2 when it fits (a 4096 x 4096
// bf16 weight is 32 MiB of the 126 MiB L2); that pass reads it "evict first".
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint4 ld_u4_policy(const void* ptr, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr), "l"(policy));
  return v;
}

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
  griddep_wait();
  uint32_t m2 = 0;  // two running maxima of bf16 magnitude bits, one per half
  const uint64_t pol = l2_policy_evict_last();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  // eight 16-byte loads in flight per thread
  for (; i + 7 * stride < n_vec; i += 8 * stride) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = ld_u4_policy(x + i + u * stride, pol);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      m2 = __vmaxu2(m2, v[u].x & 0x7FFF7FFFu);
      m2 = __vmaxu2(m2, v[u].y & 0x7FFF7FFFu);
      m2 = __vmaxu2(m2, v[u].z & 0x7FFF7FFFu);
      m2 = __vmaxu2(m2, v[u].w & 0x7FFF7FFFu);
    }
  }
  for (; i < n_vec; i += stride) {
    uint4 v = ld_u4_policy(x + i, pol);
    m2 = __vmaxu2(m2, v.x & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, v.y & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, v.z & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, v.w & 0x7FFF7FFFu);
  }
  griddep_launch_dependents();
  uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
  m = block_reduce_max(m, red);
  if (threadIdx.x == 0) {
    partial[blockIdx.x] = m;
    if (counter_to_clear != nullptr && blockIdx.x == 0) *counter_to_clear = 0ull;
  }
}

// ---- packed binary32 pairs (sm_100-family f32x2 arithmetic, IEEE RN) ----
typedef unsigned long long f2;

__device__ __forceinline__ f2 pk(float a, float b) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk(f2 v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
  f2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ f2 add2(f2 a, f2 b) {
  f2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
  f2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// Packed E2M1 pair (byte) -> the two values as a binary32 pair (exact).
__device__ __forceinline__ f2 e2m1x2_to_f2(uint32_t byte) {
  uint32_t h;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h) : "r"(byte));
  float lo, hi;
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
      : "=f"(lo), "=f"(hi) : "r"(h));
  return pk(lo, hi);
}

__device__ __forceinline__ uint32_t pack4(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
  return __byte_perm(__byte_perm(b0, b1, 0x0040u), __byte_perm(b2, b3, 0x0040u), 0x5410u);
}

// E2M1 codes of two values from the IEEE binary32 quotients x / eff.
__device__ __forceinline__ uint32_t exact_pair(float x0, float x1, float eff) {
  return cvt_e2m1x2(fmaxf(fminf(__fdiv_rn(x1, eff), 6.0f), -6.0f), fmaxf(fminf(__fdiv_rn(x0, eff), 6.0f), -6.0f));
}

// Non-negative E4M3 byte -> binary32 by the hardware E4M3 -> f16 conversion
// (every E4M3 value is exact in f16, and f16 -> binary32 is exact).
__device__ __forceinline__ float e4m3_value(uint32_t b) {
  float f;
  asm("{\n\t.reg .b16 e, lo, hi;\n\t.reg .b32 h;\n\tcvt.u16.u32 e, %1;\n\tcvt.rn.f16x2.e4m3x2 h, e;\n\t"
      "mov.b32 {lo, hi}, h;\n\tcvt.f32.f16 %0, lo;\n\t}"
      : "=f"(f) : "r"(b));
  return f;
}

// One candidate scale for a block of 16 values, given negated (nx2[j] =
// -elements 2j, 2j+1); eff = value(scale) * ts, bmax = max |x|.  Returns the
// block SSE and the 16 signed codes packed 8 per word (element 0 in the lowest
// nibble).  Signed values go through every step: round-to-nearest is
// symmetric, so each code's magnitude and each squared error equal those of
// |x|, and the conversion sets the code's sign bit from the quotient's sign.
// The negated form keeps that sign right for x = -0, whose quotient must stay
// -0: a sum of zeros of opposite signs rounds to +0, so the correction below
// is arranged so that for a zero x every sum it forms has two zeros of x's
// sign.
//
// Codes: RN(x / eff) for every element by Markstein's correction (P.
// Markstein, "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Develop. 34(1), 1990): with y = RN(1 / eff) (the
// IEEE reciprocal) and q = RN(x * y), the residual r = x - q * eff is exact in
// one fused step and RN(q + r * y) is the correctly rounded quotient, as long
// as nothing overflows or underflows.  Here q = RN((-x) * (-y)), the residual
// is taken as RN(q * eff - x) and the quotient as RN(q - that * y).  That is three packed operations per
// pair for every element and no data-dependent branch (quotients that land on
// an E2M1 rounding midpoint are common, since x and eff often share small
// factors, and a per-warp fallback for them cost more than the whole path).
// A block whose eff is outside the guarded range takes IEEE divisions; a
// quotient too small to be normal encodes as a zero code either way.
// Errors: d = RN(value * eff - x) (one fused step; the negative of
// RN(x - value * eff), so every square is the same), then
// a_j = RN(d_j^2 + RN(d_j+8^2)), b_j = a_j + a_j+4, c_j = b_j + b_j+2,
// SSE = c_0 + c_1.  A product only ever feeds the addend of an explicit fma,
// so no compiler contraction can change the rounding.
__device__ __forceinline__ float cand(const f2 (&nx2)[8], float bmax, float eff, uint32_t (&codes)[2]) {
  uint32_t bl[8];
  const f2 eff2 = pk(eff, eff);
  if (eff == 0.0f) {  // every code is a zero carrying the sign of its element
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float n0, n1;
      upk(nx2[j], n0, n1);
      bl[j] = cvt_e2m1x2(__fmul_rn(n1, -0.0f), __fmul_rn(n0, -0.0f));
    }
  } else {
    const float y = __frcp_rn(eff);
    if (eff >= 0x1p-100f && __fmul_rn(bmax, y) < 0x1p100f) {
      const f2 ny2 = pk(-y, -y);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const f2 q = mul2(nx2[j], ny2);                                   // RN(x * y)
        float q0, q1;
        upk(fma2(fma2(q, eff2, nx2[j]), ny2, q), q0, q1);  // RN(x / eff), satfinite to +-6 below
        bl[j] = cvt_e2m1x2(q1, q0);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float n0, n1;
        upk(nx2[j], n0, n1);
        bl[j] = exact_pair(-n0, -n1, eff);
      }
    }
  }
  codes[0] = pack4(bl[0], bl[1], bl[2], bl[3]);
  codes[1] = pack4(bl[4], bl[5], bl[6], bl[7]);
  f2 d[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) d[j] = fma2(e2m1x2_to_f2(bl[j]), eff2, nx2[j]);
  f2 a[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) a[j] = fma2(d[j], d[j], mul2(d[4 + j], d[4 + j]));  // (a_2j, a_2j+1)
  const f2 b0 = add2(a[0], a[2]), b1 = add2(a[1], a[3]);                           // (b_0,b_1), (b_2,b_3)
  float c0, c1;
  upk(add2(b0, b1), c0, c1);
  return __fadd_rn(c0, c1);
}

// One tile of the MMA scale layout (128 rows x 4 blocks of 16): thread i
// quantises blocks (i/4, i%4) and (i/4 + 64, i%4) from their 16 bf16 values
// v[h] (h = 0, 1; ok[h] false for padding), writes codes, logical scales and
// choices, stages the tile's 512 scale bytes in `stage` and writes them with
// one coalesced store (padding rows and columns become 0 there).  All threads
// of the CTA call it (it synchronises the CTA when scales_mma is written).
template <bool kFos>
__device__ __forceinline__ void quantize_tile(const uint4 (&v)[2][2], const bool (&ok)[2], const int64_t (&rr)[2],
                                              int64_t t, int c, int ri, int ci, int kb, float ts, bool fast6,
                                              float yts, uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                                              uint8_t* __restrict__ scales_mma, uint8_t* __restrict__ choice,
                                              uint8_t* stage, uint32_t& n_m4) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t s = 0;
    if (ok[h]) {
      const uint32_t w[8] = {v[h][0].x, v[h][0].y, v[h][0].z, v[h][0].w,
                             v[h][1].x, v[h][1].y, v[h][1].z, v[h][1].w};
      f2 nx2[8];  // negated values, elements (2j, 2j+1): adding 2^31 toggles the sign bit
      uint32_t m2 = 0;  // largest magnitude bits, per half
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        nx2[j] = pk(__uint_as_float(w[j] * 65536u + 0x80000000u), __uint_as_float((w[j] & 0xFFFF0000u) ^ 0x80000000u));
        m2 = __vmaxu2(m2, w[j] & 0x7FFF7FFFu);
      }
      const float bmax = __uint_as_float(max(m2 & 0xFFFFu, m2 >> 16) << 16);
      // s6 = E4M3(RN(RN(amax_block / 6) / ts)): each division by Markstein's
      // correction (RN(1/6) is a constant, yts = RN(1 / ts)); a block maximum
      // too small for RN(bmax / 6) to be normal, or a tensor scale outside
      // the normal range, takes the IEEE divisions.
      uint32_t s6;
      if (__builtin_expect(fast6 && (bmax >= 0x1p-120f || bmax == 0.0f), 1)) {
        constexpr float kInv6 = 1.0f / 6.0f;  // RN(1/6)
        float q = __fmul_rn(bmax, kInv6);
        q = __fmaf_rn(__fmaf_rn(q, -6.0f, bmax), kInv6, q);
        float u = __fmul_rn(q, yts);
        u = __fmaf_rn(__fmaf_rn(u, -ts, q), yts, u);
        s6 = cvt_e4m3x2(0.0f, u) & 0xFFu;
      } else {
        s6 = cvt_e4m3x2(0.0f, __fdiv_rn(__fdiv_rn(bmax, 6.0f), ts)) & 0xFFu;
      }
      const float s6v = e4m3_value(s6);
      uint32_t cw[2];
      const float sse6 = cand(nx2, bmax, __fmul_rn(s6v, ts), cw);
      s = s6;
      const int64_t blk = rr[h] * kb + c;
      if (kFos) {
        const uint32_t s4 = cvt_e4m3x2(0.0f, __fmul_rn(s6v, 1.5f)) & 0xFFu;
        bool m4 = false;
        if (s4 != s6) {  // equal scales tie, and a tie keeps M=6
          uint32_t cw4[2];
          const float sse4 = cand(nx2, bmax, __fmul_rn(e4m3_value(s4), ts), cw4);
          m4 = sse4 < sse6;
          if (m4) {
            cw[0] = cw4[0];
            cw[1] = cw4[1];
            s = s4;
            ++n_m4;
          }
        }
        if (choice != nullptr) choice[blk] = m4 ? 1 : 0;
      }
      *reinterpret_cast<uint2*>(codes + 8 * blk) = make_uint2(cw[0], cw[1]);
      if (scales != nullptr) scales[blk] = (uint8_t)s;
    }
    if (scales_mma != nullptr) {
      const int r = ri + 64 * h;  // row inside the tile
      stage[(r & 31) * 16 + (r >> 5) * 4 + ci] = (uint8_t)s;
    }
  }
  if (scales_mma != nullptr) {
    __syncthreads();
    if (threadIdx.x < kScaleTileBytes / 16)
      reinterpret_cast<uint4*>(scales_mma + t * kScaleTileBytes)[threadIdx.x] =
          reinterpret_cast<const uint4*>(stage)[threadIdx.x];
  }
}

// Four CTAs per SM for the M=6-only pass (61 registers: 12 % faster on
// 1024 x 4096 activations than three), three for FourOverSix (four would spill).
template <bool kFos>
__global__ void __launch_bounds__(kThreads, kFos ? 3 : 4)
quant_kernel(const uint4* __restrict__ x, int64_t rows, int64_t K, const uint32_t* __restrict__ partial,
             int n_partial, float divisor, uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
             uint8_t* __restrict__ scales_mma, float* __restrict__ ts_out, uint8_t* __restrict__ choice,
             unsigned long long* __restrict__ m4_count, unsigned int* __restrict__ status) {
  __shared__ uint32_t red[kThreads / 32];
  griddep_wait();  // the partials come from the amax kernel just before
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
  // the corrected divisions of s6 need ts, and so RN(1 / ts), in the normal range
  const bool fast6 = ts >= 0x1p-126f && ts <= 0x1p126f;
  const float yts = fast6 ? __frcp_rn(ts) : 0.0f;

  // Work unit: one tile of the MMA scale layout, 128 rows x 4 blocks of 16
  // (64 K positions); thread i of the CTA takes blocks (i/4, i%4) and
  // (i/4 + 64, i%4), so a warp reads 8 rows x 128 contiguous bytes and the
  // tile's 512 scale bytes are staged in shared memory and written as one
  // coalesced 512-byte store (padding rows and columns become 0 there).
  const int kb = (int)(K >> 4);
  const int ct = (kb + 3) >> 2;
  const int64_t tiles_r = (rows + 127) >> 7;
  const int64_t ntiles = tiles_r * ct;
  const int ri = threadIdx.x >> 2, ci = threadIdx.x & 3;
  __shared__ __align__(16) uint8_t stage[2][kScaleTileBytes];
  uint32_t n_m4 = 0;
  const uint64_t pol = l2_policy_evict_first();
  int buf = 0;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, buf ^= 1) {
    const int64_t tr = t / ct;
    const int tc = (int)(t - tr * ct);
    const int c = tc * 4 + ci;
    int64_t rr[2];
    bool ok[2];
    uint4 v[2][2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // both blocks' loads go out first
      rr[h] = tr * 128 + ri + 64 * h;
      ok[h] = rr[h] < rows && c < kb;
      if (ok[h]) {
        const uint4* p = x + rr[h] * (K >> 3) + 2 * c;
        v[h][0] = ld_u4_policy(p, pol);
        v[h][1] = ld_u4_policy(p + 1, pol);
      }
    }
quantize_tile<kFos>(v, ok, rr, t, c, ri, ci, kb, ts, fast6, yts, codes, scales, scales_mma, choice, stage[buf],
                        n_m4);
  }
  griddep_launch_dependents();
  if (kFos && m4_count != nullptr) {
    n_m4 = __reduce_add_sync(0xffffffffu, n_m4);
    if ((threadIdx.x & 31) == 0 && n_m4) atomicAdd(m4_count, (unsigned long long)n_m4);
  }
}

// The single-launch form, for a cooperative launch (every CTA resident at
// once): each CTA reads its tiles once -- keeping the first `resident` of
// them in shared memory -- and publishes its partial maximum; after one
// grid-wide barrier every CTA folds the partials into the tensor scale and
// quantises its tiles, the resident ones straight from shared memory.  Same
// arithmetic and results as amax_partial_kernel + quant_kernel.
template <bool kFos>
__global__ void __launch_bounds__(kThreads, 3)
quant_fused_kernel(const uint4* __restrict__ x, int64_t rows, int64_t K, uint32_t* __restrict__ partial,
                   float divisor, uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                   uint8_t* __restrict__ scales_mma, float* __restrict__ ts_out, uint8_t* __restrict__ choice,
                   unsigned long long* __restrict__ m4_count, int resident, unsigned int* __restrict__ status) {
  extern __shared__ uint4 xs[];  // [resident][2 blocks][2 pieces][kThreads]
  __shared__ uint32_t red[kThreads / 32];
  __shared__ __align__(16) uint8_t stage[2][kScaleTileBytes];
  const int kb = (int)(K >> 4);
  const int ct = (kb + 3) >> 2;
  const int64_t ntiles = ((rows + 127) >> 7) * ct;
  const int ri = threadIdx.x >> 2, ci = threadIdx.x & 3;
  auto tile_at = [&](int64_t t, int& c, int64_t (&rr)[2], bool (&ok)[2]) {
    const int64_t tr = t / ct;
    c = (int)(t - tr * ct) * 4 + ci;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      rr[h] = tr * 128 + ri + 64 * h;
      ok[h] = rr[h] < rows && c < kb;
    }
  };
  // ---- phase 1: read every tile once, the largest |x| of this CTA's ----
  const uint64_t keep = l2_policy_evict_last();  // tiles read again in phase 2 should hit L2
  uint32_t m2 = 0;
  int slot = 0;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++slot) {
    int c;
    int64_t rr[2];
    bool ok[2];
    tile_at(t, c, rr, ok);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint4 v[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
      if (ok[h]) {
        const uint4* p = x + rr[h] * (K >> 3) + 2 * c;
        v[0] = ld_u4_policy(p, keep);
        v[1] = ld_u4_policy(p + 1, keep);
#pragma unroll
        for (int j = 0; j < 2; ++j)
          m2 = __vmaxu2(__vmaxu2(m2, v[j].x & 0x7FFF7FFFu),
                        __vmaxu2(__vmaxu2(v[j].y & 0x7FFF7FFFu, v[j].z & 0x7FFF7FFFu), v[j].w & 0x7FFF7FFFu));
      }
      if (slot < resident) {
        xs[((slot * 2 + h) * 2 + 0) * kThreads + threadIdx.x] = v[0];
        xs[((slot * 2 + h) * 2 + 1) * kThreads + threadIdx.x] = v[1];
      }
    }
  }
  uint32_t am = block_reduce_max(max(m2 & 0xFFFFu, m2 >> 16), red);
  if (threadIdx.x == 0) {
    partial[blockIdx.x] = am;
    if (kFos && m4_count != nullptr && blockIdx.x == 0) *m4_count = 0ull;
  }
  cooperative_groups::this_grid().sync();  // every partial is in (and m4_count cleared)
  // ---- phase 2: the tensor scale, then the tiles ----
  am = 0;
  for (int i = threadIdx.x; i < (int)gridDim.x; i += blockDim.x) am = max(am, partial[i]);
  am = block_reduce_max(am, red);
  if (am >= 0x7F80u) {  // Inf or NaN somewhere in the tensor
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(status, kStatusNonfinite);
    return;
  }
  const float amax = __uint_as_float(am << 16);
  const float ts = amax == 0.0f ? 1.0f : __fdiv_rn(amax, divisor);
  if (blockIdx.x == 0 && threadIdx.x == 0) *ts_out = ts;
  // the corrected divisions of s6 need ts, and so RN(1 / ts), in the normal range
  const bool fast6 = ts >= 0x1p-126f && ts <= 0x1p126f;
  const float yts = fast6 ? __frcp_rn(ts) : 0.0f;
  const uint64_t once = l2_policy_evict_first();
  uint32_t n_m4 = 0;
  int buf = 0;
  slot = 0;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++slot, buf ^= 1) {
    int c;
    int64_t rr[2];
    bool ok[2];
    tile_at(t, c, rr, ok);
    uint4 v[2][2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (slot < resident) {
        v[h][0] = xs[((slot * 2 + h) * 2 + 0) * kThreads + threadIdx.x];
        v[h][1] = xs[((slot * 2 + h) * 2 + 1) * kThreads + threadIdx.x];
      } else if (ok[h]) {
        const uint4* p = x + rr[h] * (K >> 3) + 2 * c;
        v[h][0] = ld_u4_policy(p, once);
        v[h][1] = ld_u4_policy(p + 1, once);
      }
    }
    quantize_tile<kFos>(v, ok, rr, t, c, ri, ci, kb, ts, fast6, yts, codes, scales, scales_mma, choice, stage[buf],
                        n_m4);
  }
  if (kFos && m4_count != nullptr) {
    n_m4 = __reduce_add_sync(0xffffffffu, n_m4);
    if ((threadIdx.x & 31) == 0 && n_m4) atomicAdd(m4_count, (unsigned long long)n_m4);
  }
}

constexpr int kTileBytes = 2 * 2 * kThreads * 16;  // one tile's bf16 values in shared memory (16 KB)
constexpr int kMaxResident = 4;                      // tiles per CTA kept in shared memory (64 KB)

// Off by default: on GB300 the two-launch form measured faster (the
// quantiser is arithmetic-bound, and the single launch serialises the read,
// the grid barrier and the arithmetic that two launches overlap).
std::atomic<bool> g_single_launch{false};

}  // namespace

size_t quant_workspace_bytes() { return kMaxAmaxPartials * sizeof(uint32_t); }

void quantize_set_single_launch(bool on) { g_single_launch.store(on, std::memory_order_relaxed); }
bool quantize_get_single_launch() { return g_single_launch.load(std::memory_order_relaxed); }

namespace {

// The single-launch quantiser: cudaErrorNotSupported when no cooperative
// grid can be formed (the caller then uses the two-launch form).
cudaError_t launch_quantize_fused(const void* x, int64_t rows, int64_t K, float divisor, bool fos, uint8_t* codes,
                                  uint8_t* scales, uint8_t* scales_mma, float* ts, uint8_t* choice,
                                  unsigned long long* m4_count, uint32_t* partial, unsigned int* status, int num_sms,
                                  cudaStream_t stream) {
  const int64_t ntiles = ((rows + 127) / 128) * ((K / 16 + 3) / 4);
  int resident = (int)std::min<int64_t>(kMaxResident, (ntiles + 3 * num_sms - 1) / (3 * (int64_t)num_sms));
  resident = std::max(resident, 1);
  const size_t smem = (size_t)resident * kTileBytes;
  auto kern = fos ? quant_fused_kernel<true> : quant_fused_kernel<false>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  int per_sm = 0;
  if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem)) != cudaSuccess) return err;
  if (per_sm < 1) return cudaErrorNotSupported;
  const int grid = (int)std::min<int64_t>({ntiles, (int64_t)per_sm * num_sms, (int64_t)kMaxAmaxPartials});
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::max(grid, 1));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<const uint4*>(x), rows, K, partial, divisor, codes, scales,
                            scales_mma, ts, choice, fos ? m4_count : (unsigned long long*)nullptr, resident, status);
}

}  // namespace

cudaError_t launch_quantize(const void* x, int64_t rows, int64_t K, float divisor, bool fos,
                            uint8_t* codes, uint8_t* scales, uint8_t* scales_mma, float* ts,
                            uint8_t* choice, unsigned long long* m4_count, void* workspace,
                            unsigned int* status, int num_sms, cudaStream_t stream) {
  if (quantize_get_single_launch()) {
    const cudaError_t err = launch_quantize_fused(x, rows, K, divisor, fos, codes, scales, scales_mma, ts, choice,
                                                  m4_count, static_cast<uint32_t*>(workspace), status, num_sms,
                                                  stream);
    if (err != cudaErrorNotSupported) return err;
  }
  const int64_t n_vec = rows * K / 8;  // 16-byte vectors of bf16
  int g1 = (int)std::min<int64_t>((n_vec + kThreads * 4 - 1) / (kThreads * 4), (int64_t)num_sms * 4);
  g1 = std::max(1, std::min(g1, kMaxAmaxPartials));
  uint32_t* partial = static_cast<uint32_t*>(workspace);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(g1);
  cudaError_t err = cudaLaunchKernelEx(&cfg, amax_partial_kernel, static_cast<const uint4*>(x), n_vec, partial,
                                       fos ? m4_count : (unsigned long long*)nullptr);
  if (err != cudaSuccess) return err;
  const int64_t ntiles = ((rows + 127) / 128) * ((K / 16 + 3) / 4);
  int g2 = (int)std::min<int64_t>(ntiles, (int64_t)num_sms * 8);
  cfg.gridDim = dim3(std::max(g2, 1));
  if (fos)
    return cudaLaunchKernelEx(&cfg, quant_kernel<true>, static_cast<const uint4*>(x), rows, K,
                              (const uint32_t*)partial, g1, divisor, codes, scales, scales_mma, ts, choice,
                              m4_count, status);
  return cudaLaunchKernelEx(&cfg, quant_kernel<false>, static_cast<const uint4*>(x), rows, K,
                            (const uint32_t*)partial, g1, divisor, codes, scales, scales_mma, ts,
                            (uint8_t*)nullptr, (unsigned long long*)nullptr, status);
}

}  // namespace nvfp4
