// common.cuh -- device helpers shared by the NVFP4 kernels (sm_103a).
//
// Number-format conversions use the hardware cvt instructions by name; the
// bit-level decoders below follow the E2M1 / E4M3 definitions (sign, exponent,
// mantissa, bias).  Nothing here is shared with the CPU oracle.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "nvfp4.h"

namespace nvfp4 {

// Bits of the device status word (see nvfp4_get_device_status).
constexpr unsigned kStatusNonfinite = 1u;
constexpr unsigned kStatusTimeout = 2u;

constexpr int kScaleTileRows = 128;   // MMA scale tiling: 128 rows x 4 scales
constexpr int kScaleTileCols = 4;
constexpr int kScaleTileBytes = 512;

// Byte offset of logical scale (r, c) in the MMA tiling, `ct` = number of
// 4-column tiles per row tile = ceil(K/64).
__host__ __device__ __forceinline__ int64_t scale_mma_offset(int64_t r, int64_t c, int64_t ct) {
  return ((r >> 7) * ct + (c >> 2)) * kScaleTileBytes + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (c & 3);
}

// ------------------------------------------------------------ conversions ---

// Two binary32 values -> packed E4M3 pair, round to nearest even, saturating.
// hi goes to bits 15:8, lo to bits 7:0.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two binary32 values -> packed E2M1 pair (hi nibble, lo nibble), round to
// nearest even, saturating.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float hi, float lo) {
  uint32_t r;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u32.u8 %0, t;\n}"
      : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Non-negative E4M3 byte -> binary32 (exact).  Exponent field 0 is subnormal
// (m * 2^-9); otherwise 2^(e-7) * (1 + m/8).
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  uint32_t e = (b >> 3) & 15u, m = b & 7u;
  return e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : (float)m * 0x1p-9f;
}

// E2M1 magnitude code (0..7) -> binary32: 0, 0.5 for exponent field 0,
// otherwise 2^(e-1) * (1 + m/2).
__device__ __forceinline__ float e2m1_mag_to_f32(uint32_t m) {
  return m < 2u ? (float)m * 0.5f : __uint_as_float((m << 22) + (126u << 23));
}

// silu(g) * u = g / (1 + e^-g) * u in binary32 with the fast exponential and
// division intrinsics (relative error a few units in 2^-22 for |g| < 20; for
// g < -87 the quotient's divisor exceeds 2^126 and the result is 0, the
// limit).  Shared by the fused gate/up epilogue and the separate kernel, so
// both give the same bits for the same G and U.
__device__ __forceinline__ float silu_mul(float g, float u) {
  return __fmul_rn(__fdividef(g, __fadd_rn(1.0f, __expf(-g))), u);
}

// Programmatic dependent launch (kernels are launched with
// cudaLaunchAttributeProgrammaticStreamSerialization): griddep_wait() blocks
// until the previous grid in the stream has completed and its writes are
// visible; griddep_launch_dependents() lets the next grid start launching
// (it still waits for this grid to complete before reading its results).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

}  // namespace nvfp4
