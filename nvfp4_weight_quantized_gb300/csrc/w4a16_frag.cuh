// w4a16_frag.cuh -- register-level pieces shared by the W4A16 kernels that
// multiply f16 operands with warp-level MMAs: E2M1 code bytes to f16 pairs
// scaled by their E4M3 block scale, the m16n8k16 MMA, bf16 activations to
// f16 times a power of two, and shared-memory accessors.
//
// Exactness: the hardware E2M1x2 -> f16x2 conversion gives the two weights of
// a code byte exactly, and value * scale (at most 6 significant bits, within
// [2^-10, 2688]) is exact in f16, so one f16x2 multiply per byte dequantises
// without rounding.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace nvfp4 {
namespace w4a16 {

__device__ __forceinline__ uint32_t f16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// E4M3 block scale -> the same value in both halves of an f16x2 (exact: every
// E4M3 value, subnormals included, is a normal f16).
__device__ __forceinline__ uint32_t scale_f16x2(uint32_t sbyte) {
  uint32_t s;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(s) : "r"(sbyte * 0x101u));
  return s;
}

// 4 code bytes -> 4 f16x2 words of value * scale; word i holds the two
// elements of byte i (low nibble in the low half).
__device__ __forceinline__ void dequant4(uint32_t v, uint32_t s2, uint32_t* out) {
  uint32_t o0, o1, o2, o3;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o0), "=r"(o1), "=r"(o2), "=r"(o3)
      : "r"(v));
  out[0] = f16x2_mul(o0, s2);
  out[1] = f16x2_mul(o1, s2);
  out[2] = f16x2_mul(o2, s2);
  out[3] = f16x2_mul(o3, s2);
}

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 2^e as binary32 for -126 <= e <= 127.
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

// bf16 pair * c -> f16 pair (c a power of two; the binary32 products are exact).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w, float c) {
  const float lo = __fmul_rn(__uint_as_float(w << 16), c);
  const float hi = __fmul_rn(__uint_as_float(w & 0xFFFF0000u), c);
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint32_t lds8(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}

}  // namespace w4a16
}  // namespace nvfp4
