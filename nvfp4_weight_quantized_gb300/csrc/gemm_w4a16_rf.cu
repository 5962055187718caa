// gemm_w4a16_rf.cu -- decode-sized W4A16: bf16 activations x NVFP4 weights,
// weights dequantised in the register file and multiplied with warp-level
// MMAs, fp32 accumulation in registers.
//
// The small-M path of "SOAR 2026 Recap ...", section "1. Quantization and
// GEMM dispatch" (W4A16 below the crossover).  At M <= 64 tokens the GEMM is
// a weight stream: 0.5625 bytes of codes and scales per weight, each weight
// used M times.  A tcgen05.mma of K = 16 (bf16) takes at least ~70-110 SM
// cycles to issue whatever its N, so with N = M tokens it would cost more
// than streaming the weights; a register-level m16n8k16 MMA instead costs
// 2 cycles of the SM's tensor pipe per 16 x 8 x 16 tile and needs no TMEM
// round trip for the dequantised operand.
//
// One CTA = 128 weight rows x a K slice x all tokens (up to 64):
//   * warp 8 streams, per 256-wide K stage, the 128 x 128 code bytes (TMA,
//     128-byte swizzle: rows of 128 bytes keep the copy engine's request
//     count per byte low), the stage's four 512-byte MMA-tiled scale tiles
//     (one bulk copy) and four X[tokens, 64] tiles (TMA, 128-byte swizzle)
//     into a ring of stages;
//   * warps 0-7 each own 16 weight rows.  Thread (g, t) of a warp dequantises
//     rows g and g+8, K positions [16t, 16t+16) of the chunk -- exactly one
//     16-element scale block -- so the operand layout of m16n8k16 is met by
//     permuting which K positions each MMA step sees (the same permutation
//     for the weights and for X, so the sum is unchanged): step j takes code
//     bytes 8t+2j and 8t+2j+1, i.e. K = 16t+4j .. 16t+4j+3;
//   * E2M1 bits are moved into bf16 bit positions (value * 2^-126 exactly,
//     the subnormal range encodes 0.5) and one bf16x2 multiply by
//     value(scale) * 2^119 gives value * scale * 2^-7, exact in bf16;
//   * split K runs across a thread-block cluster (up to 8 CTAs) and the fp32
//     partial tiles are summed in rank order through distributed shared
//     memory (each CTA sums one slice, with all its remote loads in flight
//     together); 2^7 * ts is applied on the way out.
// Every mbarrier wait is bounded; launched with programmatic dependent launch
// (set-up overlaps the previous kernel, inputs are read after the wait).
#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace nvfp4 {

namespace {

using namespace sm100;

constexpr int BM = 128;                 // weight rows per CTA
constexpr int kChunkK = 64;             // K per MMA group (4 steps of 16)
constexpr int kStageK = 256;            // K per pipeline stage: 128 code bytes per row
constexpr int kChunksPerStage = kStageK / kChunkK;
constexpr int kRowWarps = 8;            // 16 rows each
// Compute warps: kRowWarps * SPLIT, SPLIT warps per row group taking the
// chunks of a stage in turn (SPLIT = 2 for narrow token tiles, where more
// warps hide more latency; 1 for wide ones, whose accumulators need the
// registers); the producer warp comes last.
template <int SPLIT>
struct Warps {
  static constexpr int kCompute = kRowWarps * SPLIT;
  static constexpr int kProducer = kCompute;
  static constexpr int kThreads = 32 * (kCompute + 1);
};
constexpr int split_for(int nt) { return nt <= 2 ? 2 : 1; }
constexpr int kCodeBytes = BM * kStageK / 2;             // 16 KB per stage
constexpr int kSfBytes = kChunksPerStage * kScaleTileBytes;  // 2 KB per stage
constexpr int kMaxTok = 64;
constexpr int kMaxCluster = 8;
constexpr int kMaxStages = 8;
constexpr int kRedStride = BM + 4;      // fp32 words per token row of the partial tile

struct Layout {
  int stages, n_tok;                     // n_tok: tokens per CTA, multiple of 8
  uint32_t x_tile, x_stage, codes_off, sf_off, bar_off, total;
  __host__ __device__ Layout(int st, int nt) : stages(st), n_tok(nt) {
    x_tile = ((uint32_t)nt * 128u + 1023u) & ~1023u;     // one chunk: swizzled rows of 128 bytes
    x_stage = kChunksPerStage * x_tile;
    codes_off = (uint32_t)st * x_stage;                  // X tiles first (1024-aligned)
    sf_off = codes_off + (uint32_t)st * kCodeBytes;
    uint32_t region = sf_off + (uint32_t)st * kSfBytes;
    const uint32_t red = (uint32_t)nt * kRedStride * 4u;  // partial tile, reuses the stages
    if (region < red) region = red;
    bar_off = (region + 7u) & ~7u;
    total = bar_off + 2u * kMaxStages * 8u + 1024u;       // + alignment slack
  }
};

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// value(E4M3 byte) * 2^119 as a replicated bf16 pair.  The byte shifted to
// binary32 bits 27:20 is value * 2^-120 for every finite E4M3 (the subnormal
// scales land on binary32 subnormals, zero stays zero), so exact multiplies
// by 2^120 and 2^119 give the product (at most 448 * 2^119 < 2^128); it has
// at most 4 significant bits, so its upper half is the exact bf16.
__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t sbyte) {
  const float v = __fmul_rn(__fmul_rn(__uint_as_float(sbyte << 20), 0x1p120f), 0x1p119f);
  const uint32_t b = __float_as_uint(v);
  return __byte_perm(b, b, 0x3232u);
}

// prmt.b32 in its generic form: a selector nibble with bit 3 set replicates
// the sign bit of the selected byte (__byte_perm ignores that bit).
__device__ __forceinline__ uint32_t prmt_sx(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// 4 code bytes -> 4 bf16x2 words of value * scale * 2^-7; word i holds the
// two elements of byte i (low nibble in the low half).
__device__ __forceinline__ void dequant4(uint32_t v, uint32_t s2, uint32_t* out) {
  const uint32_t lo = v & 0x0F0F0F0Fu, hi = (v >> 4) & 0x0F0F0F0Fu;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    // byte 0 <- low nibble of byte i, byte 2 <- its high nibble, bytes 1 and
    // 3 <- 0 (sign replication of a byte whose top bit is clear)
    uint32_t z = prmt_sx(lo, hi, (uint32_t)(i | 0x80 | ((4 + i) << 8) | 0x8000));
    // magnitude -> bf16 bits 8:6 (exponent 1:0, top mantissa bit), sign -> 15
    z = (z * 0x1040u) & 0x81C081C0u;
    out[i] = bf16x2_mul(z, s2);
  }
}

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
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
__device__ __forceinline__ uint32_t lds8(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}

__device__ __forceinline__ void mbar_arrive_cta(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Remote (distributed shared memory) 16-byte load; not volatile, so several
// can be in flight.
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t local_saddr, uint32_t rank) {
  uint32_t remote;
  asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_saddr), "r"(rank));
  float4 v;
  asm("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(remote));
  return v;
}

// Two CTAs per SM (registers): the 8-warp variants are held to 112
// registers, the 16-warp ones need fewer than 60 anyway.
template <int NT, bool kF32, int SPLIT = split_for(NT), typename Wp = Warps<SPLIT>>
__global__ void __launch_bounds__(Wp::kThreads, 3 - SPLIT)
w4a16_rf_kernel(const __grid_constant__ CUtensorMap tmap_codes, const __grid_constant__ CUtensorMap tmap_x,
                const uint8_t* __restrict__ smma, const float* __restrict__ ts_ptr, int64_t M, int64_t N,
                int64_t K, int stages, int stages_per_split, int prefetch_w, void* __restrict__ y,
                unsigned int* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int n_tok = 8 * NT;
  const Layout L(stages, n_tok);
  uint64_t* full = reinterpret_cast<uint64_t*>(base + L.bar_off);
  uint64_t* empty = full + kMaxStages;
  const uint32_t sbase = smem_addr(base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n0 = (int64_t)blockIdx.x * BM;
  const int64_t m0 = (int64_t)blockIdx.z * n_tok;
  const int nchunk = (int)(K / kChunkK);
  const int nstage_total = (nchunk + kChunksPerStage - 1) / kChunksPerStage;
  const int st_begin = blockIdx.y * stages_per_split;
  const int nst = max(0, min(st_begin + stages_per_split, nstage_total) - st_begin);
  const int64_t ct = K / 64;

  constexpr int kComputeWarps = Wp::kCompute, kProducerWarp = Wp::kProducer, kThreads = Wp::kThreads;
  if (threadIdx.x == kProducerWarp * 32) {
    prefetch_tmap(&tmap_codes);
    prefetch_tmap(&tmap_x);
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kComputeWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  // The next kernel in the stream may start its own prologue now: it waits
  // (griddepcontrol.wait) for this grid to finish before it touches data.
  const bool producer = threadIdx.x == kProducerWarp * 32;
  const uint8_t* sf_row_tile = smma + (n0 / 128) * ct * kScaleTileBytes;
  auto chunks_of = [&](int i) { return min(kChunksPerStage, nchunk - kChunksPerStage * (st_begin + i)); };
  auto arm = [&](int i) {  // the code box is always 128 x 128 bytes (zero fill past K)
    mbar_arrive_expect_tx(&full[i % stages], (uint32_t)(kCodeBytes + chunks_of(i) * (kScaleTileBytes + n_tok * 128)));
  };
  auto load_w = [&](int i) {  // codes and scales of stage i
    const int s = i % stages, st = st_begin + i;
    tma_load_2d(base + L.codes_off + s * kCodeBytes, &tmap_codes, st * (kStageK / 2), (int)n0, &full[s]);
    bulk_load(base + L.sf_off + s * kSfBytes, sf_row_tile + (int64_t)kChunksPerStage * st * kScaleTileBytes,
              (uint32_t)chunks_of(i) * kScaleTileBytes, &full[s]);
  };
  auto load_x = [&](int i) {
    const int s = i % stages, st = st_begin + i, chunks = chunks_of(i);
    for (int q = 0; q < chunks; ++q)
      tma_load_2d(base + s * L.x_stage + q * L.x_tile, &tmap_x, st * kStageK + q * kChunkK, (int)m0, &full[s]);
  };
  const int first = min(nst, stages);
  // Weights declared static (nvfp4_set_weight_prefetch) are requested before
  // the wait on the previous kernel, overlapping its epilogue.
  if (producer && prefetch_w) {
    for (int i = 0; i < first; ++i) arm(i);
    for (int i = 0; i < first; ++i) load_w(i);
  }
  griddep_wait();  // X (and possibly W) come from earlier kernels; Y may be read by them

  bool failed = false;
  float acc[NT][4];
#pragma unroll
  for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      // initial fill: the weight stream (the HBM reads) goes out first, then
      // the activation tiles (small, mostly L2 hits)
      if (!prefetch_w) {
        for (int i = 0; i < first; ++i) arm(i);
        for (int i = 0; i < first; ++i) load_w(i);
      }
      for (int i = 0; i < first; ++i) load_x(i);
      for (int i = first; i < nst; ++i) {
        if (!mbar_wait(&empty[i % stages], (uint32_t)(i / stages - 1) & 1u)) {
          failed = true;
          break;
        }
        arm(i);
        load_w(i);
        load_x(i);
      }
      // every copy must have landed before the stages are reused for the
      // reduction or the CTA exits
      for (int i = max(0, nst - stages); i < nst && !failed; ++i)
        if (!mbar_wait(&full[i % stages], (uint32_t)(i / stages) & 1u)) failed = true;
      if (failed) atomicOr(status, kStatusTimeout);
    }
  } else {
    const int g = lane >> 2, t = lane & 3;
    const int r0 = (warp % kRowWarps) * 16 + g, r1 = r0 + 8;
    const int par = warp / kRowWarps;  // this warp takes the chunks q of a stage with q % SPLIT == par
    // code rows: 128 bytes each, 16-byte unit u stored at u ^ (row & 7); both
    // rows of this thread have (row & 7) == g.  Chunk q, thread t reads bytes
    // 32q + 8t .. +8: unit 2q + t/2, half t & 1.
    const uint32_t crow0 = (uint32_t)(r0 * 128 + (t & 1) * 8), crow1 = (uint32_t)(r1 * 128 + (t & 1) * 8);
    const uint32_t sf0 = (uint32_t)((r0 & 31) * 16 + (r0 >> 5) * 4 + t);
    const uint32_t sf1 = (uint32_t)((r1 & 31) * 16 + (r1 >> 5) * 4 + t);
    // X tile: token row r at r * 128, 16-byte unit u stored at u ^ (r & 7)
    uint32_t xoff[NT][2];
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      const int tok = 8 * i + g;
      xoff[i][0] = (uint32_t)(tok * 128 + (((2 * t) ^ (tok & 7)) << 4));
      xoff[i][1] = (uint32_t)(tok * 128 + (((2 * t + 1) ^ (tok & 7)) << 4));
    }
    // with a single token tile the MMA chain alternates between two
    // accumulators so consecutive MMAs do not wait on each other
    float acc2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int i = 0; i < nst; ++i) {
      const int s = i % stages;
      if (!mbar_wait(&full[s], (uint32_t)(i / stages) & 1u)) {
        failed = true;
        break;
      }
      const int chunks = min(kChunksPerStage, nchunk - kChunksPerStage * (st_begin + i));
      const uint32_t cb = sbase + L.codes_off + s * kCodeBytes;
      const uint32_t sb = sbase + L.sf_off + s * kSfBytes;
      for (int q = par; q < chunks; q += SPLIT) {
        const uint32_t unit = (uint32_t)((((2 * q + (t >> 1)) ^ g)) << 4);
        const uint2 w0 = lds64(cb + crow0 + unit), w1 = lds64(cb + crow1 + unit);
        const uint32_t s0 = scale_bf16x2(lds8(sb + q * kScaleTileBytes + sf0));
        const uint32_t s1 = scale_bf16x2(lds8(sb + q * kScaleTileBytes + sf1));
        uint32_t a0[8], a1[8];  // bf16x2 of bytes 8t .. 8t+7 of rows r0 and r1
        dequant4(w0.x, s0, a0);
        dequant4(w0.y, s0, a0 + 4);
        dequant4(w1.x, s1, a1);
        dequant4(w1.y, s1, a1 + 4);
        const uint32_t xb = sbase + s * L.x_stage + q * L.x_tile;
        if (NT == 1) {
          const uint4 xa = lds128(xb + xoff[0][0]), xc = lds128(xb + xoff[0][1]);
          mma_16816(acc[0], a0[0], a1[0], a0[1], a1[1], xa.x, xa.y);
          mma_16816(acc2, a0[2], a1[2], a0[3], a1[3], xa.z, xa.w);
          mma_16816(acc[0], a0[4], a1[4], a0[5], a1[5], xc.x, xc.y);
          mma_16816(acc2, a0[6], a1[6], a0[7], a1[7], xc.z, xc.w);
        } else {
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            const uint4 xa = lds128(xb + xoff[n][0]), xc = lds128(xb + xoff[n][1]);
            mma_16816(acc[n], a0[0], a1[0], a0[1], a1[1], xa.x, xa.y);
            mma_16816(acc[n], a0[2], a1[2], a0[3], a1[3], xa.z, xa.w);
            mma_16816(acc[n], a0[4], a1[4], a0[5], a1[5], xc.x, xc.y);
            mma_16816(acc[n], a0[6], a1[6], a0[7], a1[7], xc.z, xc.w);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_cta(&empty[s]);
    }
    if (NT == 1) {
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[0][e] += acc2[e];
    }
    if (failed && lane == 0) atomicOr(status, kStatusTimeout);
  }
  // The next kernel in the stream may start its prologue now (it waits for
  // this grid to finish before it touches data).  Triggered here rather than
  // at the start: CTAs of the next grid placed early would double up on the
  // SMs this grid leaves idle.
  griddep_launch_dependents();

  // ---------------- epilogue: partial tile -> cluster reduction -> Y ----------------
  __syncthreads();  // all stages consumed and landed: reuse them for the partial tile
  float* red = reinterpret_cast<float*>(base);  // [n_tok][kRedStride]
  // the odd-chunk warps store their partial sums, the even-chunk warps of the
  // same rows add theirs (a named barrier over the compute warps in between)
  for (int ph = SPLIT - 1; ph >= 0; --ph) {
    if (warp < kComputeWarps && warp / kRowWarps == ph) {
      const int g = lane >> 2, t = lane & 3;
      const int r0 = (warp % kRowWarps) * 16 + g;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const int tok = 8 * n + 2 * t;
        float* p0 = red + tok * kRedStride + r0;
        float* p1 = p0 + kRedStride;
        if (ph == SPLIT - 1) {
          p0[0] = acc[n][0];
          p1[0] = acc[n][1];
          p0[8] = acc[n][2];
          p1[8] = acc[n][3];
        } else {
          p0[0] += acc[n][0];
          p1[0] += acc[n][1];
          p0[8] += acc[n][2];
          p1[8] += acc[n][3];
        }
      }
    }
    if (SPLIT > 1 && ph > 0 && warp < kComputeWarps)
      asm volatile("bar.sync 1, %0;" ::"n"(kComputeWarps * 32) : "memory");
  }
  cluster_sync_all();
  {
    // CTA `rank` sums groups of 4 consecutive rows of one token over the
    // cluster (in rank order) and stores them; all remote loads of a group
    // are issued before the sum
    const uint32_t ks = gridDim.y, rank = cluster_ctarank();
    const int64_t m_valid = (M - m0) < n_tok ? (M - m0) : (int64_t)n_tok;
    const int ngrp = (int)m_valid * (BM / 4);
    const int lo = (int)((rank * (uint32_t)ngrp) / ks), hi = (int)(((rank + 1) * (uint32_t)ngrp) / ks);
    const float alpha = __fmul_rn(*ts_ptr, 128.0f);
    for (int i = lo + threadIdx.x; i < hi; i += kThreads) {
      const int tk = i / (BM / 4), row = 4 * (i % (BM / 4));
      const uint32_t a = sbase + (uint32_t)(tk * kRedStride + row) * 4u;
      float4 v[kMaxCluster];
#pragma unroll
      for (int q = 0; q < kMaxCluster; ++q)
        if (q < (int)ks) v[q] = ld_dsmem_f4(a, (uint32_t)q);
      float4 sum = v[0];
#pragma unroll
      for (int q = 1; q < kMaxCluster; ++q)
        if (q < (int)ks) {
          sum.x += v[q].x;
          sum.y += v[q].y;
          sum.z += v[q].z;
          sum.w += v[q].w;
        }
      const int64_t m = m0 + tk, n = n0 + row;
      const float o[4] = {sum.x * alpha, sum.y * alpha, sum.z * alpha, sum.w * alpha};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (n + e < N) {
          if (kF32) static_cast<float*>(y)[m * N + n + e] = o[e];
          else static_cast<__nv_bfloat16*>(y)[m * N + n + e] = __float2bfloat16_rn(o[e]);
        }
      }
    }
  }
  // peers may still be reading this CTA's partial tile; the loads they wait
  // for have returned before their stores, so no ordering is needed here
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(p);
    return (EncodeTiledFn) nullptr;
  }();
  return fn;
}

bool make_map(CUtensorMap* map, CUtensorMapDataType dt, uint32_t elem_bytes, const void* base, uint64_t rows,
              uint64_t cols, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swz) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * elem_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NT>
void* kernel_for(bool f32, int* threads) {
  *threads = Warps<split_for(NT)>::kThreads;
  return f32 ? (void*)w4a16_rf_kernel<NT, true> : (void*)w4a16_rf_kernel<NT, false>;
}

}  // namespace

int w4a16_rf_max_tokens() { return kMaxTok; }

// Split of the K stages over a cluster.  Graph-timed sweeps of the split on
// GB300 (decode and MLP weight shapes, M = 1 and 16) picked these; other
// shapes use the rule below.
struct SplitEntry {
  int64_t N, K;
  int ks;
};
constexpr SplitEntry kMeasuredSplit[] = {{4096, 4096, 8}, {11008, 4096, 3}, {22016, 4096, 2}, {4096, 11008, 4}};

// Rule: minimise the per-SM share of stage units (CTAs per SM times stages
// per CTA) plus a per-wave cost of about three stages (start-up latency and
// the cluster reduction), with `resident` (1 or 2) CTAs per SM at a time;
// ties go to the larger split (more SMs, co-resident CTAs hide each other's
// latency).  The measured entries assume two resident CTAs.
void w4a16_rf_split(int64_t N, int64_t K, int64_t tiles, int nstage, int num_sms, int resident, int* ks_out,
                    int* sps_out) {
  int best_ks = 1, best_sps = nstage;
  int64_t best_cost = INT64_MAX;
  resident = std::max(1, std::min(resident, 2));
  for (const SplitEntry& e : kMeasuredSplit)
    if (e.N == N && e.K == K && tiles == (N + BM - 1) / BM && resident == 2) {
      best_ks = std::min(e.ks, nstage);
      best_sps = (nstage + best_ks - 1) / best_ks;
      *ks_out = (nstage + best_sps - 1) / best_sps;
      *sps_out = best_sps;
      return;
    }
  for (int ks = 1; ks <= kMaxCluster && ks <= nstage; ++ks) {
    const int sps = (nstage + ks - 1) / ks;
    if ((nstage + sps - 1) / sps != ks) continue;  // every CTA of the cluster gets work
    const int64_t ctas = tiles * ks;
    const int64_t waves = (ctas + (int64_t)resident * num_sms - 1) / ((int64_t)resident * num_sms);
    const int64_t cost = ((ctas + num_sms - 1) / num_sms) * sps + 3 * waves;
    if (cost <= best_cost) {
      best_cost = cost;
      best_ks = ks;
      best_sps = sps;
    }
  }
  *ks_out = best_ks;
  *sps_out = best_sps;
}

cudaError_t launch_gemm_w4a16_rf(const void* x, int64_t M, const uint8_t* codes, const uint8_t* scales_mma,
                                 const float* ts, int64_t N, int64_t K, void* y, bool out_f32, bool prefetch_w,
                                 unsigned int* status, int num_sms, cudaStream_t stream) {
  if (M <= 0) return cudaSuccess;
  if (K % 64 != 0 || N > INT32_MAX || M > INT32_MAX) return cudaErrorNotSupported;
  const int64_t n_tok_need = std::min<int64_t>(kMaxTok, (M + 7) / 8 * 8);
  int NT = (int)(n_tok_need / 8);
  if (NT == 5) NT = 6;
  if (NT == 7) NT = 8;
  const int n_tok = 8 * NT;
  const int64_t groups = (M + n_tok - 1) / n_tok;
  if (groups > 65535) return cudaErrorNotSupported;
  const int64_t tiles = (N + BM - 1) / BM;
  const int nchunk = (int)(K / kChunkK);
  const int nstage = (nchunk + kChunksPerStage - 1) / kChunksPerStage;
  void* kern = nullptr;
  int threads = 0;
  switch (NT) {
    case 1: kern = kernel_for<1>(out_f32, &threads); break;
    case 2: kern = kernel_for<2>(out_f32, &threads); break;
    case 3: kern = kernel_for<3>(out_f32, &threads); break;
    case 4: kern = kernel_for<4>(out_f32, &threads); break;
    case 6: kern = kernel_for<6>(out_f32, &threads); break;
    default: kern = kernel_for<8>(out_f32, &threads); break;
  }
  // stages in flight: as many as the split has, within ~110 KB so that two
  // CTAs can share an SM when the registers allow it
  int max_stages = kMaxStages;
  while (max_stages > 1 && Layout(max_stages, n_tok).total > 110u * 1024u) --max_stages;
  const uint32_t smem_cap = Layout(max_stages, n_tok).total;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_cap);
  if (err != cudaSuccess) return err;
  int resident = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, kern, threads, smem_cap) != cudaSuccess)
    resident = 1;
  int ks, sps;
  w4a16_rf_split(N, K, tiles * groups, nstage, num_sms, resident, &ks, &sps);
  int stages = std::max(1, std::min(sps, max_stages));
  const Layout L(stages, n_tok);
  CUtensorMap mc, mx;
  if (!make_map(&mc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, codes, (uint64_t)N, (uint64_t)K / 2, kStageK / 2, BM,
                CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, (uint64_t)M, (uint64_t)K, kChunkK, (uint32_t)n_tok,
                CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  int pf = prefetch_w ? 1 : 0;
  const uint32_t smem = L.total;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)tiles, (unsigned)ks, (unsigned)groups);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = (unsigned)ks;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  void* args[] = {(void*)&mc, (void*)&mx, (void*)&scales_mma, (void*)&ts, (void*)&M, (void*)&N, (void*)&K,
                  (void*)&stages, (void*)&sps, (void*)&pf, (void*)&y, (void*)&status};
  return cudaLaunchKernelExC(&cfg, kern, args);
}

}  // namespace nvfp4
