// gemm_w4a16.cu -- bf16 activations x NVFP4 weights, fp32 accumulation.
//
// The small-M path of "SOAR 2026 Recap ...", section "1. Quantization and
// GEMM dispatch" (W4A16 for M <= 48 on the pages' GPU).  Decode-sized GEMMs
// are bound by streaming the 0.5625 B/element weights from HBM, so the kernel
// is built around that stream:
//   * 128 weight rows per CTA (8 warps x 16), the K dimension split across a
//     thread-block cluster of up to 8 CTAs so that a 4096 x 4096 weight still
//     fills every SM;
//   * each thread streams one 16-element block (8 code bytes + 1 scale byte)
//     per row and 64-wide K chunk straight from HBM into registers, with a
//     4-deep register prefetch ring;
//   * dequantisation happens in registers and yields the A fragments of
//     mma.sync m16n8k16 directly: the E2M1 bits are placed into bf16 bit
//     positions (giving value * 2^-126 exactly) and one bf16x2 multiply by
//     value(scale) * 2^119 produces value * scale * 2^-7, exact in bf16; the
//     2^7 and the tensor scale are applied to the fp32 result;
//   * tokens are the mma N dimension (8 per tile, up to 64 per launch slice);
//   * the split-K partial tiles are reduced through distributed shared memory
//     inside the cluster (deterministic order, no global scratch).
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerCta = 128;
constexpr int kTokensPerSlice = 64;
constexpr int kPrefetch = 4;
constexpr int kMaxCluster = 8;

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// One 16-element block (8 code bytes) and its E4M3 scale -> 8 bf16x2 words,
// word i = (element 2i, element 2i+1), each = value(code) * value(scale) * 2^-7.
__device__ __forceinline__ void dequant_block(uint2 c, uint32_t sbyte, uint32_t (&out)[8]) {
  const float sf = e4m3_to_f32(sbyte) * 0x1p119f;  // exact; at most 4 significant bits
  const uint32_t sb = __float_as_uint(sf) >> 16;    // exact bf16
  const uint32_t s2 = sb | (sb << 16);
  const uint32_t w[2] = {c.x, c.y};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t v = w[h], v4 = w[h] >> 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      // low nibble of byte i -> bits 3:0, high nibble of byte i -> bits 19:16
      uint32_t z = __byte_perm(v, v4, (uint32_t)(i | (i << 4) | ((4 + i) << 8) | ((4 + i) << 12)));
      z &= 0x000F000Fu;
      // magnitude bits -> bf16 bits 8:6 (exponent 1:0, top mantissa bit), sign -> bit 15
      z = (z * 0x1040u) & 0x81C081C0u;
      out[4 * h + i] = bf16x2_mul(z, s2);
    }
  }
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ float4 ld_dsmem_f4(const float* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(remote) : "memory");
  return v;
}

template <bool kF32>
__device__ __forceinline__ void store_out(void* y, int64_t idx, float v) {
  if (kF32) static_cast<float*>(y)[idx] = v;
  else static_cast<__nv_bfloat16*>(y)[idx] = __float2bfloat16_rn(v);
}

// MT: token tiles of 8 in this launch slice (tokens m_base + blockIdx.z*64 ...).
template <int MT, bool kF32>
__global__ void __launch_bounds__(kThreads, 2)
w4a16_kernel(const __nv_bfloat16* __restrict__ x, int64_t M, int64_t m_base,
             const uint8_t* __restrict__ codes, const uint8_t* __restrict__ smma,
             const float* __restrict__ ts_ptr, int64_t N, int64_t K, int chunks_per_split,
             void* __restrict__ y) {
  extern __shared__ float4 red4[];  // [MT*8 tokens][128 rows] fp32 partial tile (split-K only)
  float* red = reinterpret_cast<float*>(red4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int64_t n0 = (int64_t)blockIdx.x * kRowsPerCta;
  const int64_t m0 = m_base + (int64_t)blockIdx.z * kTokensPerSlice;
  const int64_t r0 = n0 + warp * 16 + g, r1 = r0 + 8;
  const int64_t nchunks = K >> 6;
  const int64_t c_begin = (int64_t)blockIdx.y * chunks_per_split;
  const int64_t c_end = min(c_begin + (int64_t)chunks_per_split, nchunks);
  const int64_t ct = ((K >> 4) + 3) >> 2;
  const bool ok0 = r0 < N, ok1 = r1 < N;
  // chunk j of row r: codes bytes [32j + 8t, +8); scale (r, 4j + t) of the MMA tiling
  const uint8_t* cp0 = codes + r0 * (K >> 1) + 8 * t;
  const uint8_t* cp1 = codes + r1 * (K >> 1) + 8 * t;
  const uint8_t* sp0 = smma + ((r0 >> 7) * ct) * kScaleTileBytes + (r0 & 31) * 16 + ((r0 >> 5) & 3) * 4 + t;
  const uint8_t* sp1 = smma + ((r1 >> 7) * ct) * kScaleTileBytes + (r1 & 31) * 16 + ((r1 >> 5) & 3) * 4 + t;
  const __nv_bfloat16* xp[MT];
  bool xok[MT];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const int64_t m = m0 + 8 * mt + g;
    xok[mt] = m < M;
    xp[mt] = x + (xok[mt] ? m : 0) * K + 16 * t;
  }

  float acc[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.0f;

  uint2 rc0[kPrefetch], rc1[kPrefetch];
  uint32_t rs0[kPrefetch], rs1[kPrefetch];
#pragma unroll
  for (int u = 0; u < kPrefetch; ++u) {
    const int64_t j = c_begin + u;
    const bool live = j < c_end;
    rc0[u] = (live && ok0) ? ld_stream_u2(cp0 + 32 * j) : make_uint2(0, 0);
    rc1[u] = (live && ok1) ? ld_stream_u2(cp1 + 32 * j) : make_uint2(0, 0);
    rs0[u] = (live && ok0) ? ld_stream_u8(sp0 + j * kScaleTileBytes) : 0u;
    rs1[u] = (live && ok1) ? ld_stream_u8(sp1 + j * kScaleTileBytes) : 0u;
  }

#pragma unroll 1
  for (int64_t jb = c_begin; jb < c_end; jb += kPrefetch) {
#pragma unroll
    for (int u = 0; u < kPrefetch; ++u) {
      const int64_t j = jb + u;
      if (j < c_end) {
        uint32_t p[8], q[8];
        dequant_block(rc0[u], rs0[u], p);
        dequant_block(rc1[u], rs1[u], q);
        // refill this ring slot with chunk j + kPrefetch
        const int64_t jn = j + kPrefetch;
        const bool live = jn < c_end;
        rc0[u] = (live && ok0) ? ld_stream_u2(cp0 + 32 * jn) : make_uint2(0, 0);
        rc1[u] = (live && ok1) ? ld_stream_u2(cp1 + 32 * jn) : make_uint2(0, 0);
        rs0[u] = (live && ok0) ? ld_stream_u8(sp0 + jn * kScaleTileBytes) : 0u;
        rs1[u] = (live && ok1) ? ld_stream_u8(sp1 + jn * kScaleTileBytes) : 0u;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          uint4 xa = make_uint4(0, 0, 0, 0), xb = make_uint4(0, 0, 0, 0);
          if (xok[mt]) {
            xa = ld_cached_u4(xp[mt] + 64 * j);
            xb = ld_cached_u4(xp[mt] + 64 * j + 8);
          }
          const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            const uint32_t a[4] = {p[2 * s], q[2 * s], p[2 * s + 1], q[2 * s + 1]};
            mma_bf16(acc[mt], a, xw[2 * s], xw[2 * s + 1]);
          }
        }
      }
    }
  }

  const float alpha = __fmul_rn(*ts_ptr, 128.0f);
  if (gridDim.y == 1) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int64_t m = m0 + 8 * mt + 2 * t;
      if (m < M) {
        if (ok0) store_out<kF32>(y, m * N + r0, acc[mt][0] * alpha);
        if (ok1) store_out<kF32>(y, m * N + r1, acc[mt][2] * alpha);
      }
      if (m + 1 < M) {
        if (ok0) store_out<kF32>(y, (m + 1) * N + r0, acc[mt][1] * alpha);
        if (ok1) store_out<kF32>(y, (m + 1) * N + r1, acc[mt][3] * alpha);
      }
    }
    return;
  }

  // split-K: partial tile to shared memory, then a cluster-wide reduction in
  // which CTA `rank` sums one slice of the tile over all CTAs of the cluster.
  const int rl0 = warp * 16 + g, rl1 = rl0 + 8;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const int tk = 8 * mt + 2 * t;
    red[tk * kRowsPerCta + rl0] = acc[mt][0];
    red[(tk + 1) * kRowsPerCta + rl0] = acc[mt][1];
    red[tk * kRowsPerCta + rl1] = acc[mt][2];
    red[(tk + 1) * kRowsPerCta + rl1] = acc[mt][3];
  }
  cluster_sync_all();
  const uint32_t ks = gridDim.y;
  const uint32_t rank = cluster_ctarank();
  constexpr int kVec = MT * 8 * kRowsPerCta / 4;  // float4 elements in the tile
  const int lo = (int)((rank * (uint32_t)kVec) / ks), hi = (int)(((rank + 1) * (uint32_t)kVec) / ks);
  for (int i = lo + threadIdx.x; i < hi; i += kThreads) {
    float4 s = ld_dsmem_f4(red + 4 * i, 0);
    for (uint32_t q = 1; q < ks; ++q) {
      const float4 v = ld_dsmem_f4(red + 4 * i, q);
      s.x += v.x;
      s.y += v.y;
      s.z += v.z;
      s.w += v.w;
    }
    const int tk = (4 * i) / kRowsPerCta, nl = (4 * i) % kRowsPerCta;
    const int64_t m = m0 + tk, n = n0 + nl;
    if (m < M) {
      const float v[4] = {s.x * alpha, s.y * alpha, s.z * alpha, s.w * alpha};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (n + e < N) store_out<kF32>(y, m * N + n + e, v[e]);
    }
  }
  cluster_sync_all();
}

template <int MT, bool kF32>
cudaError_t launch_slice(const void* x, int64_t M, int64_t m_base, int64_t slices, const uint8_t* codes,
                         const uint8_t* smma, const float* ts, int64_t N, int64_t K, void* y, int num_sms,
                         cudaStream_t stream) {
  const int64_t tiles = (N + kRowsPerCta - 1) / kRowsPerCta;
  const int64_t nchunks = K / 64;
  int64_t ks = (2 * (int64_t)num_sms + tiles * slices - 1) / (tiles * slices);
  ks = std::max<int64_t>(1, std::min<int64_t>({ks, (int64_t)kMaxCluster, nchunks}));
  const int64_t cps = (nchunks + ks - 1) / ks;
  ks = (nchunks + cps - 1) / cps;
  const size_t smem = ks > 1 ? (size_t)MT * 8 * kRowsPerCta * sizeof(float) : 0;
  auto kern = w4a16_kernel<MT, kF32>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)tiles, (unsigned)ks, (unsigned)slices);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = (unsigned)ks;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<const __nv_bfloat16*>(x), M, m_base, codes, smma, ts, N,
                            K, (int)cps, y);
}

template <bool kF32>
cudaError_t launch_mt(int mt, const void* x, int64_t M, int64_t m_base, int64_t slices, const uint8_t* codes,
                      const uint8_t* smma, const float* ts, int64_t N, int64_t K, void* y, int num_sms,
                      cudaStream_t s) {
  switch (mt) {
    case 1: return launch_slice<1, kF32>(x, M, m_base, slices, codes, smma, ts, N, K, y, num_sms, s);
    case 2: return launch_slice<2, kF32>(x, M, m_base, slices, codes, smma, ts, N, K, y, num_sms, s);
    case 3: return launch_slice<3, kF32>(x, M, m_base, slices, codes, smma, ts, N, K, y, num_sms, s);
    case 4: return launch_slice<4, kF32>(x, M, m_base, slices, codes, smma, ts, N, K, y, num_sms, s);
    case 5: return launch_slice<5, kF32>(x, M, m_base, slices, codes, smma, ts, N, K, y, num_sms, s);
    case 6: return launch_slice<6, kF32>(x, M, m_base, slices, codes, smma, ts, N, K, y, num_sms, s);
    case 7: return launch_slice<7, kF32>(x, M, m_base, slices, codes, smma, ts, N, K, y, num_sms, s);
    default: return launch_slice<8, kF32>(x, M, m_base, slices, codes, smma, ts, N, K, y, num_sms, s);
  }
}

}  // namespace

cudaError_t launch_gemm_w4a16(const void* x, int64_t M, const uint8_t* codes, const uint8_t* scales_mma,
                              const float* ts, int64_t N, int64_t K, void* y, bool out_f32, int num_sms,
                              cudaStream_t stream) {
  if (M <= 0) return cudaSuccess;
  const int64_t full = M / kTokensPerSlice;
  const int64_t rem = M - full * kTokensPerSlice;
  cudaError_t err = cudaSuccess;
  if (full > 0) {
    err = out_f32 ? launch_mt<true>(8, x, M, 0, full, codes, scales_mma, ts, N, K, y, num_sms, stream)
                  : launch_mt<false>(8, x, M, 0, full, codes, scales_mma, ts, N, K, y, num_sms, stream);
    if (err != cudaSuccess) return err;
  }
  if (rem > 0) {
    const int mt = (int)((rem + 7) / 8);
    const int64_t base = full * kTokensPerSlice;
    err = out_f32 ? launch_mt<true>(mt, x, M, base, 1, codes, scales_mma, ts, N, K, y, num_sms, stream)
                  : launch_mt<false>(mt, x, M, base, 1, codes, scales_mma, ts, N, K, y, num_sms, stream);
  }
  return err;
}

}  // namespace nvfp4
