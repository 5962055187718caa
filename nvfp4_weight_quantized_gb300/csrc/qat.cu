// qat.cu -- the backward pass of an NVFP4-forward linear layer (quantisation-
// aware training with the straight-through estimator).
//
// "SOAR 2026 Recap ...", section "3. EAGLE-3 speculative decoding and hybrid
// architecture adaptation", paragraph "NVFP4 QAT": the forward GEMM runs in
// FP4 itself (nvfp4_gemm_w4a4 here) and the backward pass sends the
// gradients straight through the quantisers to the bf16 master weights.  For
// Y = X_hat W_hat^T that gives dX = dY W_hat and dW = dY^T X_hat, plain bf16
// GEMMs with fp32 accumulation.  Both run on this library's CTA-pair
// tensor-core kernel in its bf16 mode (tcgen05 kind::f16, launch_gemm_bf16_tn),
// which wants both operands K-major (the reduced index contiguous):
//   dX [M, K] = dY [M, N] * (W_hat^T [K, N])^T   -- reduced over N;
//   dW [N, K] = dY^T [N, M] * (X_hat^T [K, M])^T  -- reduced over M;
// so the NVFP4 operands are dequantised straight into transposed bf16
// buffers (dequant_bf16_t_kernel) and dY is transposed (transpose_t_kernel),
// rows padded with zeros to a multiple of 16 elements.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;
constexpr int kTile = 64;        // transposing kernels: 64 x 64 tiles
constexpr int kTilePitch = 72;   // bf16 per shared-memory tile row (16-byte aligned, fewer bank conflicts)

// value(code) * value(scale) is exact in binary32 (at most 2 + 4 significant
// bits); times the tensor scale rounded once; then rounded to bf16 (reading
// R18 of the design notes).  No integer-to-float conversion: the code's
// magnitude bits placed at binary32 bits 24:22 and its sign at bit 31 read as
// value(code) * 2^-126 exactly (0.5 lands in the subnormal range, and a
// negative zero code gives -0).  Its product with the E4M3 scale is exact too
// (at most 6 significant bits, none below 2^-141), and the product times
// 2^126 is exactly value(code) * value(scale).
__device__ __forceinline__ float code_bits(uint32_t code) {
  return __uint_as_float(((code & 7u) << 22) | ((code & 8u) << 28));  // value(code) * 2^-126
}

__device__ __forceinline__ float dequant_value(uint32_t code, float s, float ts) {
  return __fmul_rn(__fmul_rn(__fmul_rn(code_bits(code), s), 0x1p126f), ts);
}

// packed binary32 pairs (lo in the low word)
__device__ __forceinline__ unsigned long long pack_f2(float lo, float hi) {
  unsigned long long d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ unsigned long long mul_f2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// both halves rounded to bf16 (round to nearest even): lo -> bits 15:0
__device__ __forceinline__ uint32_t bf16x2_of(unsigned long long v) {
  uint32_t d;
  asm("{\n\t.reg .f32 a, b;\n\tmov.b64 {a, b}, %1;\n\tcvt.rn.bf16x2.f32 %0, b, a;\n\t}" : "=r"(d) : "l"(v));
  return d;
}

// One 16-element block per thread and step: 8 code bytes in, 32 bytes out.
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
      __nv_bfloat162 p = __floats2bfloat162_rn(dequant_value(byte & 15u, s, ts), dequant_value(byte >> 4, s, ts));
      o[j] = *reinterpret_cast<uint32_t*>(&p);
    }
    uint4* dst = reinterpret_cast<uint4*>(out + r * K + 16 * c);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// The transposing kernels stage a tile in shared memory as bf16 pairs: word
// (c, p) holds source rows 2p and 2p + 1 of tile column c (row 2p in the low
// half), i.e. two adjacent elements of output row c.  A thread owns one row
// pair, so every shared-memory write is a whole word, and word p of row c is
// stored at p ^ swz(c) with swz(c) a multiple of 4: the 32 threads of a warp
// that write one tile column hit 32 different banks, and four consecutive
// words (one 16-byte piece of an output row) stay together.
constexpr int kPairWords = kTile / 2;  // words per staged tile row (64 source rows)

__device__ __forceinline__ uint32_t pair_lo(uint32_t a, uint32_t b) { return __byte_perm(a, b, 0x5410u); }
__device__ __forceinline__ uint32_t pair_hi(uint32_t a, uint32_t b) { return __byte_perm(a, b, 0x7632u); }

// NVFP4 [R, K] -> bf16 out^T [K, Rp] (out[k * Rp + r]), columns R .. Rp - 1
// zero; Rp % 8 == 0.  A CTA covers 64 rows x 256 K positions: thread (p, q)
// dequantises 16-element blocks 2q and 2q + 1 of rows 2p and 2p + 1 (one
// 16-byte code load per row; the 8 threads of a row pair read its 128 code
// bytes contiguously), the tile is staged transposed as described above (here
// swz(c) = 4 * ((c / 32) % 8), the block pair of tile column c), and the CTA
// writes 256 output rows of 128 bytes with 16-byte stores.
constexpr int kDqK = 256;  // K positions per CTA
__global__ void __launch_bounds__(kThreads)
dequant_bf16_t_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ smma,
                      const float* __restrict__ ts_ptr, int64_t R, int64_t K, int64_t Rp,
                      __nv_bfloat16* __restrict__ out) {
  __shared__ __align__(16) uint32_t tw[kDqK][kPairWords];
  griddep_wait();
  const float ts = *ts_ptr;
  const int64_t kb = K / 16, ct = (kb + 3) / 4;
  const int64_t r0 = (int64_t)blockIdx.x * kTile, k0 = (int64_t)blockIdx.y * kDqK;
  {
    const int q = threadIdx.x & 7, p = threadIdx.x >> 3;  // block pair, row pair of the tile
    const int64_t c = k0 / 16 + 2 * q;                     // first of the two blocks
    // codes and scales of blocks c, c + 1 of rows 2p (e = 0) and 2p + 1;
    // zero codes and scales outside the matrix give +0
    uint2 cw[2][2];
    float sc[2][2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int64_t r = r0 + 2 * p + e;
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        cw[e][blk] = make_uint2(0u, 0u);
        sc[e][blk] = 0.0f;
      }
      if (r < R && c < kb) {
        const uint8_t* row = codes + r * (K / 2) + 8 * c;
        if (c + 1 < kb && (reinterpret_cast<uintptr_t>(row) & 15) == 0) {
          const uint4 v = *reinterpret_cast<const uint4*>(row);
          cw[e][0] = make_uint2(v.x, v.y);
          cw[e][1] = make_uint2(v.z, v.w);
        } else {
          cw[e][0] = *reinterpret_cast<const uint2*>(row);
          if (c + 1 < kb) cw[e][1] = *reinterpret_cast<const uint2*>(row + 8);
        }
#pragma unroll
        for (int blk = 0; blk < 2; ++blk)
          if (c + blk < kb) sc[e][blk] = e4m3_to_f32(smma[scale_mma_offset(r, c + blk, ct)]);
      }
    }
    // word j of block blk: the bf16 pair (row 2p, row 2p + 1) of element j,
    // both values formed as in dequant_value by packed binary32 multiplies
    // (each lane rounded as the scalar multiply rounds it)
    uint32_t w[2][16];
    const unsigned long long two126 = pack_f2(0x1p126f, 0x1p126f), ts2 = pack_f2(ts, ts);
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      const unsigned long long s2 = pack_f2(sc[0][blk], sc[1][blk]);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t n0 = ((j < 8 ? cw[0][blk].x : cw[0][blk].y) >> (4 * (j & 7))) & 15u;
        const uint32_t n1 = ((j < 8 ? cw[1][blk].x : cw[1][blk].y) >> (4 * (j & 7))) & 15u;
        const unsigned long long v2 = pack_f2(code_bits(n0), code_bits(n1));
        w[blk][j] = bf16x2_of(mul_f2(mul_f2(mul_f2(v2, s2), two126), ts2));
      }
    }
    const int sw = p ^ (4 * q);  // tile columns 32q .. 32q + 31
#pragma unroll
    for (int blk = 0; blk < 2; ++blk)
#pragma unroll
      for (int j = 0; j < 16; ++j) tw[32 * q + 16 * blk + j][sw] = w[blk][j];
  }
  __syncthreads();
#pragma unroll
  for (int pass = 0; pass < kDqK / 32; ++pass) {
    const int cc = (threadIdx.x >> 3) + 32 * pass, u = threadIdx.x & 7;
    const int64_t k = k0 + cc, r = r0 + 8 * u;
    if (k < K && r < Rp)
      *reinterpret_cast<uint4*>(out + k * Rp + r) =
          *reinterpret_cast<const uint4*>(&tw[cc][4 * (u ^ ((cc >> 5) & 7))]);
  }
}

// bf16 [rows, cols] (row pitch `spitch`) -> dst^T [cols, rows_p]
// (dst[c * rows_p + r]), rows rows .. rows_p - 1 zero; rows_p % 8 == 0.  A CTA
// covers a 64 x 64 tile: thread (p, v) reads the 8 columns 8v .. 8v + 7 of
// rows 2p and 2p + 1 (16-byte loads when the rows are 16-byte aligned and the
// piece lies inside the source), the tile is staged transposed as described
// above, and the CTA writes 64 output rows of 128 bytes with 16-byte stores.
__global__ void __launch_bounds__(kThreads)
transpose_t_kernel(const __nv_bfloat16* __restrict__ src, int64_t rows, int64_t cols, int64_t spitch,
                   __nv_bfloat16* __restrict__ dst, int64_t rows_p) {
  __shared__ __align__(16) uint32_t tw[kTile][kPairWords];
  griddep_wait();
  const int64_t r0 = (int64_t)blockIdx.x * kTile, c0 = (int64_t)blockIdx.y * kTile;
  const bool vec = (spitch & 7) == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0;
  {
    const int p = threadIdx.x >> 3, v = threadIdx.x & 7;  // row pair, 8-column piece
    const int64_t c = c0 + 8 * v;
    uint4 x[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int64_t r = r0 + 2 * p + e;
      x[e] = make_uint4(0u, 0u, 0u, 0u);
      if (r < rows) {
        const __nv_bfloat16* row = src + r * spitch;
        if (vec && c + 8 <= cols) {
          x[e] = *reinterpret_cast<const uint4*>(row + c);
        } else {
          uint16_t hv[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) hv[j] = c + j < cols ? reinterpret_cast<const uint16_t*>(row)[c + j] : 0;
          x[e] = make_uint4(hv[0] | ((uint32_t)hv[1] << 16), hv[2] | ((uint32_t)hv[3] << 16),
                            hv[4] | ((uint32_t)hv[5] << 16), hv[6] | ((uint32_t)hv[7] << 16));
        }
      }
    }
    const uint32_t a[4] = {x[0].x, x[0].y, x[0].z, x[0].w}, bb[4] = {x[1].x, x[1].y, x[1].z, x[1].w};
    const int sw = p ^ (4 * v);  // tile columns 8v .. 8v + 7: swz = 4 * (column >> 3) = 4v
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      tw[8 * v + 2 * j][sw] = pair_lo(a[j], bb[j]);
      tw[8 * v + 2 * j + 1][sw] = pair_hi(a[j], bb[j]);
    }
  }
  __syncthreads();
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    const int cc = (threadIdx.x >> 3) + 32 * pass, u = threadIdx.x & 7;
    const int64_t c = c0 + cc, r = r0 + 8 * u;
    if (c < cols && r < rows_p)
      *reinterpret_cast<uint4*>(dst + c * rows_p + r) = *reinterpret_cast<const uint4*>(&tw[cc][4 * (u ^ (cc >> 3))]);
  }
}

// bf16 [rows, cols] (row pitch `spitch`) -> dst [rows, cols_p], columns
// cols .. cols_p - 1 zero; cols_p % 8 == 0 (a copy of dY whose rows are not
// 16-byte aligned).  64 x 64 tiles through shared memory.
__global__ void __launch_bounds__(kThreads)
pad_copy_bf16_kernel(const __nv_bfloat16* __restrict__ src, int64_t rows, int64_t cols, int64_t spitch,
                     __nv_bfloat16* __restrict__ dst, int64_t cols_p) {
  __shared__ __align__(16) __nv_bfloat16 tile[kTile][kTilePitch];
  griddep_wait();
  const int64_t r0 = (int64_t)blockIdx.x * kTile, c0 = (int64_t)blockIdx.y * kTile;
  const __nv_bfloat16 zero = __float2bfloat16_rn(0.0f);
  for (int i = threadIdx.x; i < kTile * kTile; i += kThreads) {  // coalesced along the source row
    const int rl = i >> 6, cl = i & 63;
    const int64_t r = r0 + rl, c = c0 + cl;
    tile[rl][cl] = (r < rows && c < cols) ? src[r * spitch + c] : zero;
  }
  __syncthreads();
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {  // 64 destination rows of 8 16-byte pieces
    const int rl = (threadIdx.x >> 3) + 32 * pass, v8 = threadIdx.x & 7;
    const int64_t r = r0 + rl, c = c0 + 8 * v8;
    if (r < rows && c < cols_p)
      *reinterpret_cast<uint4*>(dst + r * cols_p + c) = *reinterpret_cast<const uint4*>(&tile[rl][8 * v8]);
  }
}

cudaLaunchConfig_t pdl_config(dim3 grid, cudaStream_t stream, cudaLaunchAttribute* attr) {
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

int64_t round16(int64_t v) { return (v + 15) / 16 * 16; }

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace

cudaError_t launch_dequant_bf16(const uint8_t* codes, const uint8_t* scales_mma, const float* ts, int64_t R,
                                int64_t K, void* out, int num_sms, cudaStream_t stream) {
  if (R <= 0) return cudaSuccess;
  const int64_t nblk = R * (K / 16);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(
      dim3((unsigned)std::min<int64_t>((nblk + kThreads - 1) / kThreads, (int64_t)num_sms * 8)), stream, attr);
  return cudaLaunchKernelEx(&cfg, dequant_bf16_kernel, codes, scales_mma, ts, R, K,
                            static_cast<__nv_bfloat16*>(out));
}

size_t qat_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  // W_hat^T [K, Np], X_hat^T [K, Mp], dY^T [N, Mp], and a padded dY [M, Np]
  // when its rows are not 16-byte aligned
  const size_t Mp = (size_t)round16(M), Np = (size_t)round16(N), k = (size_t)K, m = (size_t)M;
  return align256(k * Np * 2) + align256(k * Mp * 2) + align256((size_t)N * Mp * 2) +
         (N % 8 != 0 ? align256(m * Np * 2) : 0);
}

cudaError_t qat_backward(const void* dy, int64_t M, const uint8_t* w_codes, const uint8_t* w_smma, const float* w_ts,
                         int64_t N, int64_t K, const uint8_t* a_codes, const uint8_t* a_smma, const float* a_ts,
                         void* dx, void* dw, void* workspace, unsigned int* status, cudaStream_t stream) {
  if (M <= 0 || (dx == nullptr && dw == nullptr)) return cudaSuccess;
  const int64_t Mp = round16(M), Np = round16(N);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto* wt = reinterpret_cast<__nv_bfloat16*>(ws);                          // W_hat^T [K, Np]
  auto* xt = reinterpret_cast<__nv_bfloat16*>(ws + align256((size_t)K * Np * 2));  // X_hat^T [K, Mp]
  auto* dyt = reinterpret_cast<__nv_bfloat16*>(reinterpret_cast<uint8_t*>(xt) + align256((size_t)K * Mp * 2));
  auto* dyp = reinterpret_cast<__nv_bfloat16*>(reinterpret_cast<uint8_t*>(dyt) + align256((size_t)N * Mp * 2));
  const auto* dyb = static_cast<const __nv_bfloat16*>(dy);
  cudaLaunchAttribute attr[1];
  cudaError_t err;
  if (dx != nullptr) {
    // dX [M, K] = dY [M, N] . W_hat^T [K, N]: reduced over N
    cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)((N + kTile - 1) / kTile), (unsigned)((K + kDqK - 1) / kDqK)),
                                        stream, attr);
    if ((err = cudaLaunchKernelEx(&cfg, dequant_bf16_t_kernel, w_codes, w_smma, w_ts, N, K, Np, wt)) != cudaSuccess)
      return err;
    const __nv_bfloat16* a = dyb;
    int64_t pitch = N;
    if (N % 8 != 0) {  // rows of dY are not 16-byte aligned: a zero-padded copy [M, Np]
      cfg = pdl_config(dim3((unsigned)((M + kTile - 1) / kTile), (unsigned)((N + kTile - 1) / kTile)), stream, attr);
      if ((err = cudaLaunchKernelEx(&cfg, pad_copy_bf16_kernel, dyb, M, N, N, dyp, Np)) != cudaSuccess)
        return err;
      a = dyp;
      pitch = Np;
    }
    if ((err = launch_gemm_bf16_tn(a, pitch, wt, Np, M, K, N, dx, false, status, stream)) != cudaSuccess) return err;
  }
  if (dw != nullptr) {
    // dW [N, K] = dY^T [N, Mp] . X_hat^T [K, Mp]: reduced over M
    cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)((M + kTile - 1) / kTile), (unsigned)((K + kDqK - 1) / kDqK)),
                                        stream, attr);
    if ((err = cudaLaunchKernelEx(&cfg, dequant_bf16_t_kernel, a_codes, a_smma, a_ts, M, K, Mp, xt)) != cudaSuccess)
      return err;
    cfg = pdl_config(dim3((unsigned)((M + kTile - 1) / kTile), (unsigned)((N + kTile - 1) / kTile)), stream, attr);
    if ((err = cudaLaunchKernelEx(&cfg, transpose_t_kernel, dyb, M, N, N, dyt, Mp)) != cudaSuccess)
      return err;
    if ((err = launch_gemm_bf16_tn(dyt, Mp, xt, Mp, N, K, M, dw, true, status, stream)) != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace nvfp4
