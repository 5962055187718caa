// gemm_w4a4.cu -- NVFP4 x NVFP4 GEMM on the 5th-generation tensor cores.
//
// The large-M path of "SOAR 2026 Recap ...", section "1. Quantization and GEMM
// dispatch": activations quantised online to NVFP4, then a GEMM built on the
// block-scaled FP4 tensor-core MMA itself.  On sm_103a that instruction is
// tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X: E2M1 operands packed
// two per byte, one UE4M3 scale per 16 elements along K, fp32 accumulation in
// tensor memory (TMEM).
//
// Persistent kernel, one CTA per SM, looping over 128 x BN output tiles
// (A rows = tokens, B rows = weight rows), 10 warps:
//   warp 8, one lane  -- producer: per 256-wide K stage, TMA loads of the A and
//                        B code tiles (128-byte swizzle) and bulk copies of the
//                        matching scale tiles (already in the MMA tiling);
//   warps 4-7         -- scale loaders: copy the stage's scale tiles from shared
//                        memory into TMEM with tcgen05.st (lane = tile row);
//   warp 9, one lane  -- MMA issuer: four K=64 MMAs per stage and nothing
//                        else (an MMA stream is bound by its issuer's latency);
//   warps 0-3         -- epilogue: tcgen05.ld of the accumulator, scale by
//                        ts_a * ts_w, convert, store, release the accumulator.
// BN = 256 for large M.  When M fits one tile, the narrowest weight tile
// (64, 128 or 256 rows) whose tiles fit one wave of CTAs: a skinny GEMM
// spreads over the SMs, and no SM streams a second tile after the others have
// finished (64-row tiles on W[11008, 4096] took two waves and 1.4x as long).  Every mbarrier wait is bounded; a wait that
// runs out sets the library's status word (NVFP4_ERR_TIMEOUT) and the CTA
// winds down.
#include <cuda.h>
#include <cuda_bf16.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace nvfp4 {

namespace {

using namespace sm100;

constexpr int BM = 128;             // tokens per tile (MMA M = TMEM lanes)
constexpr int BK = 256;             // FP4 elements per stage (128 bytes per row)
constexpr int kEpiWarps = 4, kSfWarps = 4;
constexpr int kProducerWarp = kEpiWarps + kSfWarps, kMmaWarp = kProducerWarp + 1;
constexpr int kThreads = 32 * (kMmaWarp + 1);
constexpr uint32_t kTmemCols = 512;
constexpr int kABytes = BM * BK / 2;                      // 16 KB
constexpr int kSfaBytes = (BK / 64) * kScaleTileBytes;    // 2 KB: 4 atoms (one per K=64 MMA)

template <int BN>
struct Cfg {
  // operand stages: 3 for the wide tile, whose epilogue also stages half an
  // output tile (32 KB) in shared memory for TMA stores; 6 for the 128-row
  // tile (a one-wave weight stream at M <= 128, bound by the copies each CTA
  // has in flight); 4 for the 64-row one
  static constexpr int kStages = BN == 256 ? 3 : BN == 128 ? 6 : 4;
  static constexpr int kYStageBytes = BN == 256 ? 2 * BM * 128 : 1024;  // two 128 x 64 bf16 boxes (unused at BN = 64)
  static constexpr int kBBytes = BN * BK / 2;
  static constexpr int kSfbTiles = (BN + 127) / 128;                        // 128-row scale tiles
  static constexpr int kSfbBytes = kSfbTiles * (BK / 64) * kScaleTileBytes;
  static constexpr uint32_t kAccCol = 0;                                    // BN fp32 columns
  static constexpr uint32_t kSfaCols = 16;                                  // 4 MMAs x 4 columns
  static constexpr uint32_t kSfbCols = 16 * kSfbTiles;                      // 4 MMAs x 4 columns per tile
  static constexpr uint32_t kSfCol = BN;                                    // per-stage scale columns
  static constexpr uint32_t kSfStageCols = kSfaCols + kSfbCols;
  static_assert(kSfCol + kStages * kSfStageCols <= kTmemCols, "TMEM budget");
  // instruction descriptor, kind::mxf4nvf4: A and B E2M1 (format code 1 in
  // bits 7-9 and 10-12), both K-major, N >> 3 in bits 17-22, scale type
  // UE4M3 (bit 23 = 0), M >> 7 in bits 27-28, scale-factor ids 0, dense
  static constexpr uint32_t kIdesc =
      (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 7) << 27);
};

template <int BN>
struct __align__(1024) Smem {
  static constexpr int kStages = Cfg<BN>::kStages;
  uint8_t ystage[Cfg<BN>::kYStageBytes];  // first: 1024-aligned for the 128-byte swizzle
  uint8_t a[kStages][kABytes];
  uint8_t b[kStages][Cfg<BN>::kBBytes];
  uint8_t sfa[kStages][kSfaBytes];
  uint8_t sfb[kStages][Cfg<BN>::kSfbBytes];
  uint64_t full[kStages];     // TMA landed
  uint64_t sf_full[kStages];  // scales in TMEM (4 loader warps)
  uint64_t empty[kStages];    // MMAs of the stage done
  uint64_t acc_full;          // tile accumulated
  uint64_t acc_free;          // epilogue drained the accumulator (4 warps)
  uint32_t tmem_base;
};

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}


// Two floats -> bf16 pair (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}


template <bool kF32>
__device__ __forceinline__ void store_row32(void* y, int64_t row_off, int64_t n, int64_t N, const uint32_t (&v)[32],
                                            float alpha, bool vec_ok) {
  if (kF32) {
    float* out = static_cast<float*>(y) + row_off + n;
    if (vec_ok && n + 32 <= N) {
#pragma unroll
      for (int i = 0; i < 32; i += 4)
        *reinterpret_cast<float4*>(out + i) =
            make_float4(__uint_as_float(v[i]) * alpha, __uint_as_float(v[i + 1]) * alpha,
                        __uint_as_float(v[i + 2]) * alpha, __uint_as_float(v[i + 3]) * alpha);
    } else {
      for (int i = 0; i < 32 && n + i < N; ++i) out[i] = __uint_as_float(v[i]) * alpha;
    }
  } else {
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(y) + row_off + n;
    if (vec_ok && n + 32 <= N) {
#pragma unroll
      for (int i = 0; i < 32; i += 8) {
        uint4 p;
        __nv_bfloat162 h0 = __floats2bfloat162_rn(__uint_as_float(v[i]) * alpha, __uint_as_float(v[i + 1]) * alpha);
        __nv_bfloat162 h1 =
            __floats2bfloat162_rn(__uint_as_float(v[i + 2]) * alpha, __uint_as_float(v[i + 3]) * alpha);
        __nv_bfloat162 h2 =
            __floats2bfloat162_rn(__uint_as_float(v[i + 4]) * alpha, __uint_as_float(v[i + 5]) * alpha);
        __nv_bfloat162 h3 =
            __floats2bfloat162_rn(__uint_as_float(v[i + 6]) * alpha, __uint_as_float(v[i + 7]) * alpha);
        p.x = *reinterpret_cast<uint32_t*>(&h0);
        p.y = *reinterpret_cast<uint32_t*>(&h1);
        p.z = *reinterpret_cast<uint32_t*>(&h2);
        p.w = *reinterpret_cast<uint32_t*>(&h3);
        *reinterpret_cast<uint4*>(out + i) = p;
      }
    } else {
      for (int i = 0; i < 32 && n + i < N; ++i) out[i] = __float2bfloat16_rn(__uint_as_float(v[i]) * alpha);
    }
  }
}

// kGateUp (BN = 256, bf16 output): W is a gated-MLP input projection [2F, K]
// (rows [0, F) gate, [F, 2F) up, F % 128 == 0); a tile covers 128 features,
// its B stage holding their gate rows (first 128 rows) and up rows (last 128),
// so accumulator column j < 128 of a row holds G[m, f0 + j] and column 128 + j
// holds U[m, f0 + j], and the epilogue writes silu(G) * U for F features.
template <int BN, bool kF32, bool kGateUp = false>
__global__ void __launch_bounds__(kThreads, 1)
w4a4_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
            const __grid_constant__ CUtensorMap tmap_y, int tma_store, const uint8_t* __restrict__ a_smma, const uint8_t* __restrict__ b_smma,
            const float* __restrict__ a_ts, const float* __restrict__ b_ts, int64_t M, int64_t N, int64_t K,
            void* __restrict__ y, unsigned int* __restrict__ status) {
  using C = Cfg<BN>;
  constexpr int kStages = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  Smem<BN>& sm = *reinterpret_cast<Smem<BN>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kb64 = (int)(K / 64);                 // 64-wide K blocks = scale column tiles per row tile
  const int kt = (kb64 + 3) / 4;                  // K stages per tile
  const int64_t b_row_tiles = (N + 127) / 128;    // row tiles present in the weight scale tiling
  static_assert(!kGateUp || (BN == 256 && !kF32), "gate/up epilogue: 256-row tiles, bf16 output");
  const int64_t F = N / 2;                        // features of a gate/up weight
  const int64_t m_tiles = (M + BM - 1) / BM, n_tiles = kGateUp ? F / 128 : (N + BN - 1) / BN;
  const int64_t n_work = m_tiles * n_tiles;

  if (warp == kProducerWarp && lane == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.sf_full[s], kSfWarps);
      mbar_init(&sm.empty[s], 1);
    }
    mbar_init(&sm.acc_full, 1);
    mbar_init(&sm.acc_free, kEpiWarps);
    fence_mbar_init();
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
  }
  if (warp == 0) tmem_alloc(&sm.tmem_base, kTmemCols);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = sm.tmem_base;
  bool failed = false;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      // ---------------- producer ----------------
      griddep_wait();  // inputs may be written by the previous kernel in the stream
      int g = 0;       // stage counter across this CTA's tiles
      for (int64_t w = blockIdx.x; w < n_work && !failed; w += gridDim.x) {
        const int64_t m_tile = w / n_tiles, n_tile = w - m_tile * n_tiles;
        const int64_t n0 = n_tile * (kGateUp ? 128 : BN);
        const int64_t sfb_left = b_row_tiles - n0 / 128;
        const int nsfb = kGateUp ? 2 : sfb_left < C::kSfbTiles ? (int)sfb_left : C::kSfbTiles;
        for (int ks = 0; ks < kt; ++ks, ++g) {
          const int s = g % kStages;
          if (g >= kStages && !mbar_wait(&sm.empty[s], (uint32_t)(g / kStages - 1) & 1u)) {
            failed = true;
            break;
          }
          const int kk_n = min(4, kb64 - 4 * ks);
          const uint32_t sf_bytes = (uint32_t)kk_n * kScaleTileBytes;
          mbar_arrive_expect_tx(&sm.full[s], kABytes + C::kBBytes + sf_bytes * (1 + nsfb));
          tma_load_2d(sm.a[s], &tmap_a, ks * (BK / 2), (int)(m_tile * BM), &sm.full[s]);
          tma_load_2d(sm.b[s], &tmap_b, ks * (BK / 2), (int)n0, &sm.full[s]);
          if (kGateUp)  // the up rows of the same features (the B map's box is 128 rows here)
            tma_load_2d(sm.b[s] + C::kBBytes / 2, &tmap_b, ks * (BK / 2), (int)(F + n0), &sm.full[s]);
          bulk_load(sm.sfa[s], a_smma + (m_tile * kb64 + 4 * ks) * kScaleTileBytes, sf_bytes, &sm.full[s]);
          for (int rt = 0; rt < nsfb; ++rt) {
            // scale tile of B rows 128 rt ..: the next weight row tile, or for
            // gate/up the up rows' tile F / 128 further on
            const int64_t bt = kGateUp ? (n0 + F * rt) / 128 : n0 / 128 + rt;
            bulk_load(sm.sfb[s] + rt * (BK / 64) * kScaleTileBytes, b_smma + (bt * kb64 + 4 * ks) * kScaleTileBytes,
                      sf_bytes, &sm.full[s]);
          }
        }
      }
      // let every load this thread issued land before the CTA can exit
      for (int i = max(0, g - kStages); i < g && !failed; ++i)
        if (!mbar_wait(&sm.full[i % kStages], (uint32_t)(i / kStages) & 1u)) failed = true;
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      int g = 0, t = 0;
      for (int64_t w = blockIdx.x; w < n_work && !failed; w += gridDim.x, ++t) {
        const int64_t n0 = (w % n_tiles) * BN;
        // rows of a 64-wide tile that starts in the upper half of a 128-row
        // scale tile sit in TMEM columns 2-3 of each 4-column group
        const uint32_t sfb_sub = (BN == 64 && (n0 & 127) == 64) ? 2u : 0u;
        if (t > 0 && !mbar_wait(&sm.acc_free, (uint32_t)(t - 1) & 1u)) {
          failed = true;
          break;
        }
        fence_after_sync();
        for (int ks = 0; ks < kt; ++ks, ++g) {
          const int s = g % kStages;
          if (!mbar_wait(&sm.sf_full[s], (uint32_t)(g / kStages) & 1u)) {
            failed = true;
            break;
          }
          fence_after_sync();
          const int kk_n = min(4, kb64 - 4 * ks);
          const uint32_t sfa_t = tmem + C::kSfCol + C::kSfStageCols * s;
          const uint32_t sfb_t = sfa_t + C::kSfaCols + sfb_sub;
          const uint64_t adesc = smem_desc(smem_addr(sm.a[s]), 0, 1024, 2);
          const uint64_t bdesc = smem_desc(smem_addr(sm.b[s]), 0, 1024, 2);
          // advancing the start address by 32 bytes selects the next 64 FP4
          // elements inside the 128-byte swizzle atom; a full stage is issued
          // with constant offsets (see the pair kernel's issuer)
          if (kk_n == 4) {
            const uint32_t d = tmem + C::kAccCol, acc0 = ks != 0;
            constexpr uint32_t sb = 4 * C::kSfbTiles;
            mma_mxf4nvf4(d, adesc, bdesc, C::kIdesc, sfa_t, sfb_t, acc0);
            mma_mxf4nvf4(d, adesc + 2ull, bdesc + 2ull, C::kIdesc, sfa_t + 4, sfb_t + sb, 1u);
            mma_mxf4nvf4(d, adesc + 4ull, bdesc + 4ull, C::kIdesc, sfa_t + 8, sfb_t + 2 * sb, 1u);
            mma_mxf4nvf4(d, adesc + 6ull, bdesc + 6ull, C::kIdesc, sfa_t + 12, sfb_t + 3 * sb, 1u);
          } else {
            for (int kk = 0; kk < kk_n; ++kk)
              mma_mxf4nvf4(tmem + C::kAccCol, adesc + 2ull * kk, bdesc + 2ull * kk, C::kIdesc, sfa_t + 4 * kk,
                           sfb_t + 4 * C::kSfbTiles * kk, (ks | kk) != 0);
          }
          commit(&sm.empty[s]);
        }
        if (!failed) commit(&sm.acc_full);
      }
      griddep_launch_dependents();
    }
  } else if (warp >= kEpiWarps) {
    // ---------------- scale loaders: shared memory -> TMEM ----------------
    // Each 512-byte scale atom holds 32 chunks of 16 bytes; chunk i goes to
    // lane i of every 32-lane quarter (the layout the MMA reads: row r of the
    // tile at lane r % 32 of any quarter, column r / 32), 4 columns per atom.
    // Atom order in TMEM: A: 4 * kk; B: 16 + 4 * (kSfbTiles * kk + rt).
    const uint32_t lane_base = (uint32_t)((warp - kEpiWarps) * 32) << 16;
    int g = 0;
    for (int64_t w = blockIdx.x; w < n_work && !failed; w += gridDim.x) {
      for (int ks = 0; ks < kt; ++ks, ++g) {
        const int s = g % kStages;
        if (!mbar_wait(&sm.full[s], (uint32_t)(g / kStages) & 1u)) {
          failed = true;
          break;
        }
        // the TMEM scale slot of stage s is free once the MMAs of its previous
        // round completed (that is what empty[s] signals)
        if (g >= kStages && !mbar_wait(&sm.empty[s], (uint32_t)(g / kStages - 1) & 1u)) {
          failed = true;
          break;
        }
        const uint32_t col = tmem + lane_base + C::kSfCol + C::kSfStageCols * s;
        uint32_t r[16];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint4 v = *reinterpret_cast<const uint4*>(sm.sfa[s] + kk * kScaleTileBytes + lane * 16);
          r[4 * kk] = v.x;
          r[4 * kk + 1] = v.y;
          r[4 * kk + 2] = v.z;
          r[4 * kk + 3] = v.w;
        }
        tmem_st_x16(col, r);
#pragma unroll
        for (int h = 0; h < C::kSfbTiles * 4; h += 4) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int idx = h + q;  // = kSfbTiles * kk + rt
            const int kk = idx / C::kSfbTiles, rt = idx % C::kSfbTiles;
            const uint4 v = *reinterpret_cast<const uint4*>(sm.sfb[s] + rt * (BK / 64) * kScaleTileBytes +
                                                            kk * kScaleTileBytes + lane * 16);
            r[4 * q] = v.x;
            r[4 * q + 1] = v.y;
            r[4 * q + 2] = v.z;
            r[4 * q + 3] = v.w;
          }
          tmem_st_x16(col + C::kSfaCols + 4 * h, r);
        }
        tmem_wait_st();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.sf_full[s]);
      }
    }
  } else {
    // ---------------- epilogue (warps 0-3; TMEM lanes 32w..32w+31 = tile rows) ----------------
    griddep_wait();  // the tensor scales may come from the previous kernel in the stream
    const float alpha = __fmul_rn(*a_ts, *b_ts);
    const bool vec_ok = kF32 ? (N % 4 == 0) : (N % 8 == 0);
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    int t = 0;
    for (int64_t w = blockIdx.x; w < n_work; w += gridDim.x, ++t) {
      const int64_t m_tile = w / n_tiles, n_tile = w - m_tile * n_tiles;
      const int64_t row = m_tile * BM + warp * 32 + lane, n0 = n_tile * BN;
      // warp-uniform, since tcgen05.ld is a warp-collective instruction
      const bool ok = __all_sync(0xffffffffu, !failed && mbar_wait(&sm.acc_full, (uint32_t)t & 1u));
      if (!ok) {
        failed = true;
        break;
      }
      fence_after_sync();
      if (kGateUp) {
        // silu(G) * U for features f0 .. f0 + 127 straight into the staging
        // buffer (two 128 x 64 bf16 boxes, 128-byte swizzle), then the
        // accumulator goes back and two TMA stores (clipping rows past M)
        // write the tile -- the arithmetic of the pair kernel's gate/up
        // epilogue
        const int r = warp * 32 + lane;  // tile row = TMEM lane
        const uint32_t acc = tmem + lane_base + C::kAccCol;
        if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");  // staging buffer free
#pragma unroll 1
        for (int c2 = 0; c2 < 4; ++c2) {  // 32 features per step: chunks 2 c2, 2 c2 + 1 of 16
          uint32_t vg[32], vu[32];
          tmem_ld_32x32b_x32(acc + 32 * c2, vg);
          tmem_ld_32x32b_x32(acc + 128 + 32 * c2, vu);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int c = 2 * c2 + h;
            uint32_t p[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int j = 16 * h + 2 * i;
              p[i] = bf16x2_rn(silu_mul(__uint_as_float(vg[j]) * alpha, __uint_as_float(vu[j]) * alpha),
                               silu_mul(__uint_as_float(vg[j + 1]) * alpha, __uint_as_float(vu[j + 1]) * alpha));
            }
            uint8_t* box = sm.ystage + (c >> 2) * (BM * 128) + r * 128;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int unit = ((c & 3) * 2 + u) ^ (r & 7);
              *reinterpret_cast<uint4*>(box + unit * 16) =
                  make_uint4(p[4 * u], p[4 * u + 1], p[4 * u + 2], p[4 * u + 3]);
            }
          }
        }
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.acc_free);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
        if (threadIdx.x == 0) {
#pragma unroll
          for (int j = 0; j < 2; ++j)
            asm volatile(
                "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(&tmap_y),
                "r"((int)(n_tile * 128 + 64 * j)), "r"((int)(m_tile * BM)), "r"(smem_addr(sm.ystage + j * (BM * 128)))
                : "memory");
          asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
      } else if (BN <= 64) {
        // small tile: drain it all, hand the accumulator back, then store
        uint32_t v[BN / 32][32];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) tmem_ld_32x32b_x32(tmem + lane_base + C::kAccCol + 32 * c, v[c]);
        tmem_wait_ld();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.acc_free);
        if (row < M) {
#pragma unroll
          for (int c = 0; c < BN / 32; ++c)
            if (n0 + 32 * c < N) store_row32<kF32>(y, row * N, n0 + 32 * c, N, v[c], alpha, vec_ok);
        }
      } else if (!kF32 && BN == 256 && tma_store) {
        // wide tile, bf16: each half (128 columns) is converted into two
        // 128 x 64 bf16 boxes in shared memory (128-byte swizzle) and written
        // by TMA stores; the accumulator goes back to the MMA warp as soon as
        // its last columns are in registers, so the stores overlap the next
        // tile's MMAs.  The TMA clips rows and columns outside Y.
        const int r = warp * 32 + lane;  // tile row = TMEM lane
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
          asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");  // staging buffer free
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            const int c = 4 * half + cc;
            uint32_t v[32];
            tmem_ld_32x32b_x32(tmem + lane_base + C::kAccCol + 32 * c, v);
            tmem_wait_ld();
            if (c == BN / 32 - 1) {
              fence_before_sync();
              __syncwarp();
              if (lane == 0) mbar_arrive(&sm.acc_free);
            }
            uint8_t* box = sm.ystage + (cc >> 1) * (BM * 128) + r * 128;
#pragma unroll
            for (int u = 0; u < 4; ++u) {  // 16-byte unit (cc & 1) * 4 + u of the row, swizzled
              const uint4 p = make_uint4(
                  bf16x2_rn(__uint_as_float(v[8 * u]) * alpha, __uint_as_float(v[8 * u + 1]) * alpha),
                  bf16x2_rn(__uint_as_float(v[8 * u + 2]) * alpha, __uint_as_float(v[8 * u + 3]) * alpha),
                  bf16x2_rn(__uint_as_float(v[8 * u + 4]) * alpha, __uint_as_float(v[8 * u + 5]) * alpha),
                  bf16x2_rn(__uint_as_float(v[8 * u + 6]) * alpha, __uint_as_float(v[8 * u + 7]) * alpha));
              const int unit = ((cc & 1) * 4 + u) ^ (r & 7);
              *reinterpret_cast<uint4*>(box + unit * 16) = p;
            }
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
          if (threadIdx.x == 0) {
#pragma unroll
            for (int j = 0; j < 2; ++j)
              asm volatile(
                  "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(&tmap_y),
                  "r"((int)(n0 + 128 * half + 64 * j)), "r"((int)(m_tile * BM)),
                  "r"(smem_addr(sm.ystage + j * (BM * 128)))
                  : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tmem + lane_base + C::kAccCol + 32 * c, v);
          tmem_wait_ld();
          if (row < M && n0 + 32 * c < N) store_row32<kF32>(y, row * N, n0 + 32 * c, N, v, alpha, vec_ok);
        }
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.acc_free);
      }
    }
    if (failed && lane == 0) atomicOr(status, kStatusTimeout);
    // the output stores must be complete before the grid ends
    if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Pair kernel: the same GEMM with 256 x 256 output tiles, each computed by the
// two CTAs of a cluster with cta_group::2 MMAs (M = 256, N = 256, K = 64).
// CTA r of the pair stages A rows [m0 + 128 r, +128) and B rows
// [n0 + 128 r, +128) of every K stage in its own shared memory, so a CTA
// streams half the operand bytes of the single-CTA 128 x 256 tile for the same
// MMA work, and the MMA reads each operand byte from shared memory once.  Each
// CTA holds the A scales of its rows and the B scales of all 256 tile rows in
// its own TMEM (same columns in both), and its 128 x 256 fp32 accumulator.
//
//   producer (warp 8, each CTA): TMA of its A and B halves and the scale
//     tiles into its shared memory, signalled on its own full[s];
//   scale loaders (warps 4-7, each CTA): full[s] -> TMEM -> arrive on the
//     even CTA's sf_full[s] (8 arrivals: the stage is ready in both CTAs);
//   MMA issuer (warp 9 of the even CTA): four pair MMAs per stage, then one
//     commit that arrives on empty[s] of both CTAs; acc_full[b] likewise;
//   epilogue (warps 0-3, each CTA): drains its accumulator lanes, then
//     arrives on the even CTA's acc_free[b] (8 arrivals).  b alternates
//     between two accumulators in the bf16 mode and is 0 otherwise.
// Every CTA loads its own operand tiles (no TMA multicast); rows both CTAs of
// different pairs need are shared through L2.
constexpr int kPairStages = 5;
// The pair kernel's loads are issued by three producer warps (A rows and
// their scales; B rows; B scales): one thread waits ~130-170 cycles per
// TMA or bulk-copy issue (measured), and the MMAs of a stage take ~560.
constexpr int kProdB = kMmaWarp + 1, kProdSfb = kMmaWarp + 2;
constexpr int kPairProducers = 3;
constexpr int kPairThreads = 32 * (kProdSfb + 1);

struct __align__(1024) PairSmem {
  uint8_t ystage[2 * BM * 128];          // two 128 x 64 bf16 output boxes
  uint8_t a[kPairStages][kABytes];       // this CTA's 128 A rows x 256 K
  uint8_t b[kPairStages][kABytes];       // this CTA's 128 B rows x 256 K
  uint8_t sfa[kPairStages][kSfaBytes];   // A scales of this CTA's rows
  uint8_t sfb[kPairStages][2 * kSfaBytes];  // B scales of both 128-row halves
  uint64_t full[kPairStages];     // this CTA's loads landed
  uint64_t sf_full[kPairStages];  // even CTA: scales in TMEM in both CTAs
  uint64_t empty[kPairStages];    // MMAs of the stage done (from the even CTA)
  uint64_t acc_full[2];           // tile accumulated in accumulator b (from the even CTA)
  uint64_t acc_free[2];           // even CTA: accumulator b drained in both CTAs
  uint32_t tmem_base;
};

constexpr uint32_t kPairSfCol = 256;                  // after the 256 accumulator columns
constexpr uint32_t kPairSfStageCols = 16 + 32;        // A: 4 MMAs x 4; B: 4 MMAs x 2 halves x 4
static_assert(kPairSfCol + kPairStages * kPairSfStageCols <= kTmemCols, "TMEM budget");
// kind::mxf4nvf4, E2M1 x E2M1, K-major, N = 256, UE4M3 scales, M = 256
constexpr uint32_t kPairIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(256 >> 3) << 17) | (2u << 27);
// kind::f16 (the bf16 mode below): fp32 accumulator (bits 4-5 = 1), A and B
// bf16 (format 1 in bits 7-9 and 10-12), both K-major, N >> 3 in bits 17-22,
// M >> 4 in bits 24-28 (M = 256 across the pair), dense
constexpr uint32_t kPairIdescBf16 =
    (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(256 >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);

// kBF16: the same pipeline as a plain bf16 GEMM, Y = A B^T with A [M, Kb] and
// B [N, Kb] bf16, both K-major: a 128-byte row of a stage holds 64 bf16 (256
// FP4 elements in the NVFP4 mode), the MMAs are kind::f16 with K = 16 (32
// bytes, the same descriptor step), and there are no scale factors (the
// scale producer and loaders only pass the stage on) and no tensor scales.
// The caller passes K = 4 * Kb rounded up to 64, so that K / 64 counts the
// 16-wide MMA steps.
// kGateUp: W is a gated-MLP input projection [2F, K] (rows [0, F) gate,
// [F, 2F) up, F % 128 == 0) and the kernel writes Y[m, f] = silu(G) * U for
// F features: a tile covers 128 features, CTA 0 of the pair staging their
// gate rows and CTA 1 their up rows, so accumulator column j (< 128) of every
// row holds G[m, f0 + j] and column 128 + j holds U[m, f0 + j].
template <bool kF32, bool kGateUp = false, bool kBF16 = false>
__global__ void __launch_bounds__(kPairThreads, 1)
w4a4_pair_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                 const __grid_constant__ CUtensorMap tmap_y, int tma_store, const uint8_t* __restrict__ a_smma,
                 const uint8_t* __restrict__ b_smma, const float* __restrict__ a_ts,
                 const float* __restrict__ b_ts, int64_t M, int64_t N, int64_t K, void* __restrict__ y,
                 unsigned int* __restrict__ status) {
  constexpr int S = kPairStages;
  // The bf16 mode has no scale columns, so two 256-column accumulators fit
  // in TMEM and alternate between tiles: the epilogue drains one while the
  // MMAs fill the other.  The FP4 modes have one (columns 256-495 hold the
  // stages' scale factors).
  constexpr int kAccBufs = kBF16 ? 2 : 1;
  constexpr uint32_t kAccStride = 256;
  static_assert(kAccBufs * kAccStride <= kTmemCols && (kBF16 || kAccStride <= kPairSfCol), "TMEM budget");
  extern __shared__ uint8_t smem_raw[];
  PairSmem& sm = *reinterpret_cast<PairSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();  // CTA in the pair; CTA 0 issues the MMAs
  constexpr uint32_t lead = 0;
  constexpr uint16_t pair_mask = 3u;
  const int64_t cl = blockIdx.x / 2, ncl = gridDim.x / 2;
  const int kb64 = (int)(K / 64);
  const int kt = (kb64 + 3) / 4;
  static_assert(!kGateUp || !kF32, "gate/up epilogue: bf16 output");
  const int64_t b_row_tiles = (N + 127) / 128;
  const int64_t F = N / 2;  // features of a gate/up weight
  const int64_t n_tiles = kGateUp ? F / 128 : (N + 255) / 256;
  const int64_t n_work = ((M + 255) / 256) * n_tiles;

  if (warp == kProducerWarp && lane == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&sm.full[s], kPairProducers);
      mbar_init(&sm.sf_full[s], 2 * kSfWarps);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.acc_full[b], 1);
      mbar_init(&sm.acc_free[b], 2 * kEpiWarps);
    }
    fence_mbar_init();
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
  }
  if (warp == 0) tmem_alloc_pair(&sm.tmem_base, kTmemCols);
  fence_before_sync();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any cross-CTA arrive
  fence_after_sync();
  const uint32_t tmem = sm.tmem_base;
  bool failed = false;

  if (warp == kProducerWarp || warp == kProdB || warp == kProdSfb) {
    if (lane == 0) {
      // ---------------- producers (each CTA): A + A scales / B / B scales ----------------
      griddep_wait();
      int g = 0;
      for (int64_t w = cl; w < n_work && !failed; w += ncl) {
        const int64_t m_tile = w / n_tiles, n_tile = w - m_tile * n_tiles;
        const int64_t arow = m_tile * 256 + 128 * rank;
        const int64_t n0 = n_tile * (kGateUp ? 128 : 256);
        const int64_t brow = kGateUp ? n0 + F * rank : n0 + 128 * rank;
        // a CTA whose A (or B) rows all lie past M (N) loads nothing for them:
        // its accumulator rows (or the tile's columns from that half) are never stored
        const bool has_a = arow < M, has_b = brow < N;
        const uint32_t a_bytes = has_a ? kABytes : 0;
        const int64_t sfb_left = b_row_tiles - n0 / 128;
        const int nsfb = kBF16 ? 0 : kGateUp ? 2 : sfb_left <= 0 ? 0 : sfb_left < 2 ? (int)sfb_left : 2;
        for (int ks = 0; ks < kt; ++ks, ++g) {
          const int s = g % S;
          if (g >= S && !mbar_wait(&sm.empty[s], (uint32_t)(g / S - 1) & 1u)) {
            failed = true;
            break;
          }
          const int kk_n = min(4, kb64 - 4 * ks);
          const uint32_t sf_bytes = (uint32_t)kk_n * kScaleTileBytes;
          if (warp == kProducerWarp) {
            mbar_arrive_expect_tx(&sm.full[s], a_bytes + (has_a && !kBF16 ? sf_bytes : 0));
            if (has_a) tma_load_2d(sm.a[s], &tmap_a, ks * (BK / 2), (int)arow, &sm.full[s]);
            if (has_a && !kBF16)
              bulk_load(sm.sfa[s], a_smma + ((arow / 128) * kb64 + 4 * ks) * kScaleTileBytes, sf_bytes,
                        &sm.full[s]);
          } else if (warp == kProdB) {
            mbar_arrive_expect_tx(&sm.full[s], has_b ? kABytes : 0);
            if (has_b) tma_load_2d(sm.b[s], &tmap_b, ks * (BK / 2), (int)brow, &sm.full[s]);
          } else {
            mbar_arrive_expect_tx(&sm.full[s], sf_bytes * nsfb);
            for (int rt = 0; rt < nsfb; ++rt) {
              // B rows 128 rt .. of the MMA: the next weight row tile, or for
              // gate/up the up rows' tile F / 128 further on
              const int64_t bt = kGateUp ? (n0 + F * rt) / 128 : n0 / 128 + rt;
              bulk_load(sm.sfb[s] + rt * kSfaBytes, b_smma + (bt * kb64 + 4 * ks) * kScaleTileBytes, sf_bytes,
                        &sm.full[s]);
            }
          }
        }
      }
      if (warp == kProducerWarp) griddep_launch_dependents();
      // before the CTA may exit: this CTA's loads have landed and the pair's
      // MMAs that read them have completed
      for (int i = max(0, g - S); i < g && !failed; ++i)
        if (!mbar_wait(&sm.full[i % S], (uint32_t)(i / S) & 1u) ||
            !mbar_wait(&sm.empty[i % S], (uint32_t)(i / S) & 1u))
          failed = true;
      if (failed) atomicOr(status, kStatusTimeout);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (even CTA of each pair) ----------------
      // ring slot s and phase ph advance with the stage (no divisions); the
      // descriptors and scale columns of slot s are the slot-0 ones plus s
      // strides (a descriptor's start address is in 16-byte units)
      int s = 0, t = 0;
      uint32_t ph = 0;
      const uint64_t adesc0 = smem_desc(smem_addr(sm.a[0]), 0, 1024, 2);
      const uint64_t bdesc0 = smem_desc(smem_addr(sm.b[0]), 0, 1024, 2);
      constexpr uint64_t kDescStride = (uint64_t)(kABytes >> 4);
      static_assert(sizeof(sm.a[0]) == kABytes && sizeof(sm.b[0]) == kABytes, "stage stride");
      for (int64_t w = cl; w < n_work && !failed; w += ncl, ++t) {
        // accumulator b of tile t, its use u (two alternate in the bf16 mode)
        const int b = kAccBufs == 2 ? (t & 1) : 0, u = kAccBufs == 2 ? (t >> 1) : t;
        const uint32_t acc = tmem + kAccStride * (uint32_t)b;
        if (u > 0 && !mbar_wait(&sm.acc_free[b], (uint32_t)(u - 1) & 1u)) {
          failed = true;
          break;
        }
        fence_after_sync();
        for (int ks = 0; ks < kt; ++ks) {
          if (!mbar_wait(&sm.sf_full[s], ph)) {
            failed = true;
            break;
          }
          fence_after_sync();
          const int kk_n = min(4, kb64 - 4 * ks);
          const uint32_t sfa_t = tmem + kPairSfCol + kPairSfStageCols * (uint32_t)s;
          const uint32_t sfb_t = sfa_t + 16;
          const uint64_t adesc = adesc0 + kDescStride * (uint64_t)s;
          const uint64_t bdesc = bdesc0 + kDescStride * (uint64_t)s;
          // This thread is latency-bound: every tcgen05 instruction and barrier
          // test takes ~90 cycles to issue, against 128 cycles of tensor work
          // per pair MMA, so a full stage is issued as four MMAs with constant
          // operand offsets and one accumulate flag (per-MMA address and
          // predicate arithmetic in a rolled loop lengthened the stage period
          // by ~17 %, measured).
          const uint32_t acc0 = ks != 0;
          if (kBF16) {
            if (kk_n == 4) {
              mma_f16_pair(acc, adesc, bdesc, kPairIdescBf16, acc0);
              mma_f16_pair(acc, adesc + 2ull, bdesc + 2ull, kPairIdescBf16, 1u);
              mma_f16_pair(acc, adesc + 4ull, bdesc + 4ull, kPairIdescBf16, 1u);
              mma_f16_pair(acc, adesc + 6ull, bdesc + 6ull, kPairIdescBf16, 1u);
            } else {
              for (int kk = 0; kk < kk_n; ++kk)
                mma_f16_pair(acc, adesc + 2ull * kk, bdesc + 2ull * kk, kPairIdescBf16, (ks | kk) != 0);
            }
          } else if (kk_n == 4) {
            mma_mxf4nvf4_pair(acc, adesc, bdesc, kPairIdesc, sfa_t, sfb_t, acc0);
            mma_mxf4nvf4_pair(acc, adesc + 2ull, bdesc + 2ull, kPairIdesc, sfa_t + 4, sfb_t + 8, 1u);
            mma_mxf4nvf4_pair(acc, adesc + 4ull, bdesc + 4ull, kPairIdesc, sfa_t + 8, sfb_t + 16, 1u);
            mma_mxf4nvf4_pair(acc, adesc + 6ull, bdesc + 6ull, kPairIdesc, sfa_t + 12, sfb_t + 24, 1u);
          } else {
            for (int kk = 0; kk < kk_n; ++kk)
              mma_mxf4nvf4_pair(acc, adesc + 2ull * kk, bdesc + 2ull * kk, kPairIdesc, sfa_t + 4 * kk,
                                sfb_t + 8 * kk, (ks | kk) != 0);
          }
          commit_pair(&sm.empty[s], pair_mask);
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!failed) commit_pair(&sm.acc_full[b], pair_mask);
      }
      if (failed) atomicOr(status, kStatusTimeout);
    }
  } else if (warp >= kEpiWarps) {
    // ---------------- scale loaders (each CTA): shared memory -> TMEM ----------------
    // atom kk of A at column 4 kk; atom (kk, half rt) of B at 16 + 4 (2 kk + rt)
    const uint32_t lane_base = (uint32_t)((warp - kEpiWarps) * 32) << 16;
    int g = 0;
    for (int64_t w = cl; w < n_work && !failed; w += ncl) {
      for (int ks = 0; ks < kt; ++ks, ++g) {
        const int s = g % S;
        if (!mbar_wait(&sm.full[s], (uint32_t)(g / S) & 1u) ||
            (g >= S && !mbar_wait(&sm.empty[s], (uint32_t)(g / S - 1) & 1u))) {
          failed = true;
          break;
        }
        const uint32_t col = tmem + lane_base + kPairSfCol + kPairSfStageCols * s;
        if (!kBF16) {  // bf16 mode: no scale factors, the stage is only passed on
          uint32_t r[16];
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint4 v = *reinterpret_cast<const uint4*>(sm.sfa[s] + kk * kScaleTileBytes + lane * 16);
            r[4 * kk] = v.x;
            r[4 * kk + 1] = v.y;
            r[4 * kk + 2] = v.z;
            r[4 * kk + 3] = v.w;
          }
          tmem_st_x16(col, r);
#pragma unroll
          for (int h = 0; h < 8; h += 4) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int idx = h + q;  // = 2 kk + rt
              const int kk = idx >> 1, rt = idx & 1;
              const uint4 v =
                  *reinterpret_cast<const uint4*>(sm.sfb[s] + rt * kSfaBytes + kk * kScaleTileBytes + lane * 16);
              r[4 * q] = v.x;
              r[4 * q + 1] = v.y;
              r[4 * q + 2] = v.z;
              r[4 * q + 3] = v.w;
            }
            tmem_st_x16(col + 16 + 4 * h, r);
          }
        }
        tmem_wait_st();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(&sm.sf_full[s], lead);
      }
    }
    if (failed && lane == 0) atomicOr(status, kStatusTimeout);
  } else {
    // ---------------- epilogue (each CTA; TMEM lane = tile row) ----------------
    griddep_wait();  // the tensor scales may come from the previous kernel in the stream
    const float alpha = kBF16 ? 1.0f : __fmul_rn(*a_ts, *b_ts);
    const bool vec_ok = kF32 ? (N % 4 == 0) : (N % 8 == 0);
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const int r = warp * 32 + lane;
    int t = 0;
    for (int64_t w = cl; w < n_work; w += ncl, ++t) {
      const int64_t m_tile = w / n_tiles, n_tile = w - m_tile * n_tiles;
      const int64_t m0 = m_tile * 256 + 128 * rank, n0 = n_tile * (kGateUp ? 128 : 256);
      const int64_t row = m0 + r;
      const int b = kAccBufs == 2 ? (t & 1) : 0, u = kAccBufs == 2 ? (t >> 1) : t;
      const uint32_t acc = tmem + kAccStride * (uint32_t)b + lane_base;  // this warp's lanes of accumulator b
      const bool ok = __all_sync(0xffffffffu, !failed && mbar_wait(&sm.acc_full[b], (uint32_t)u & 1u));
      if (!ok) {
        failed = true;
        break;
      }
      fence_after_sync();
      if (kGateUp) {
        // silu(G) * U for features n0 .. n0 + 127 straight into the staging
        // buffer (two 128 x 64 bf16 boxes), then the accumulator goes back
        // and one round of TMA stores writes the tile
        if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
#pragma unroll 1
        for (int c2 = 0; c2 < 4; ++c2) {  // 32 features per step: chunks 2 c2, 2 c2 + 1 of 16
          uint32_t vg[32], vu[32];
          tmem_ld_32x32b_x32(acc + 32 * c2, vg);
          tmem_ld_32x32b_x32(acc + 128 + 32 * c2, vu);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int c = 2 * c2 + h;
            uint32_t p[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int j = 16 * h + 2 * i;
              p[i] = bf16x2_rn(silu_mul(__uint_as_float(vg[j]) * alpha, __uint_as_float(vu[j]) * alpha),
                               silu_mul(__uint_as_float(vg[j + 1]) * alpha, __uint_as_float(vu[j + 1]) * alpha));
            }
            uint8_t* box = sm.ystage + (c >> 2) * (BM * 128) + r * 128;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int unit = ((c & 3) * 2 + u) ^ (r & 7);
              *reinterpret_cast<uint4*>(box + unit * 16) =
                  make_uint4(p[4 * u], p[4 * u + 1], p[4 * u + 2], p[4 * u + 3]);
            }
          }
        }
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(&sm.acc_free[b], lead);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
        if (threadIdx.x == 0 && m0 < M) {
#pragma unroll
          for (int j = 0; j < 2; ++j)
            asm volatile(
                "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(&tmap_y),
                "r"((int)(n0 + 64 * j)), "r"((int)m0), "r"(smem_addr(sm.ystage + j * (BM * 128)))
                : "memory");
          asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
      } else if (!kF32 && tma_store) {
        // Columns 0-127 go straight to the staging buffer (two 128 x 64 bf16
        // boxes, 128-byte swizzle), columns 128-255 into registers as scaled
        // bf16 pairs; then the accumulator goes back to the MMA warp and the
        // TMA stores (which clip rows past M) overlap the next tile's MMAs.
        if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");  // staging buffer free
        uint32_t hi[8][8];
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {  // 64 columns per wait (two loads in flight): chunks 4 c4 .. 4 c4 + 3 of 16
          uint32_t v0[32], v1[32];
          tmem_ld_32x32b_x32(acc + 64 * c4, v0);
          tmem_ld_32x32b_x32(acc + 64 * c4 + 32, v1);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const int c = 4 * c4 + h;
            uint32_t p[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int j = 16 * (h & 1) + 2 * i;  // a constant once unrolled: both arrays stay in registers
              const uint32_t lo = h < 2 ? v0[j] : v1[j], hi2 = h < 2 ? v0[j + 1] : v1[j + 1];
              p[i] = bf16x2_rn(__uint_as_float(lo) * alpha, __uint_as_float(hi2) * alpha);
            }
            if (c < 8) {
              uint8_t* box = sm.ystage + (c >> 2) * (BM * 128) + r * 128;
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const int unit = ((c & 3) * 2 + u) ^ (r & 7);
                *reinterpret_cast<uint4*>(box + unit * 16) =
                    make_uint4(p[4 * u], p[4 * u + 1], p[4 * u + 2], p[4 * u + 3]);
              }
            } else {
#pragma unroll
              for (int i = 0; i < 8; ++i) hi[c - 8][i] = p[i];
            }
          }
        }
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(&sm.acc_free[b], lead);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          if (half == 1) {
            if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              uint8_t* box = sm.ystage + (c >> 2) * (BM * 128) + r * 128;
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const int unit = ((c & 3) * 2 + u) ^ (r & 7);
                *reinterpret_cast<uint4*>(box + unit * 16) =
                    make_uint4(hi[c][4 * u], hi[c][4 * u + 1], hi[c][4 * u + 2], hi[c][4 * u + 3]);
              }
            }
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
          if (threadIdx.x == 0 && m0 < M) {
#pragma unroll
            for (int j = 0; j < 2; ++j)
              if (n0 + 128 * half + 64 * j < N)
                asm volatile(
                    "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(&tmap_y),
                    "r"((int)(n0 + 128 * half + 64 * j)), "r"((int)m0), "r"(smem_addr(sm.ystage + j * (BM * 128)))
                    : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
          }
        }
      } else if (kF32 && tma_store) {
        // fp32 rows leave through the staging buffer as well: four rounds of
        // 64 columns, each two 128 x 32 fp32 boxes (128-byte rows, 128-byte
        // swizzle) written by TMA stores that clip rows and columns outside
        // Y; the accumulator goes back once the last round's columns are in
        // registers.
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
          if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
          asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");  // staging buffer free
          uint32_t v0[32], v1[32];
          tmem_ld_32x32b_x32(acc + 64 * q, v0);
          tmem_ld_32x32b_x32(acc + 64 * q + 32, v1);
          tmem_wait_ld();
          if (q == 3) {
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(&sm.acc_free[b], lead);
          }
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const uint32_t* v = j == 0 ? v0 : v1;
            uint8_t* box = sm.ystage + j * (BM * 128) + r * 128;
#pragma unroll
            for (int u = 0; u < 8; ++u)
              *reinterpret_cast<float4*>(box + ((u ^ (r & 7)) << 4)) =
                  make_float4(__uint_as_float(v[4 * u]) * alpha, __uint_as_float(v[4 * u + 1]) * alpha,
                              __uint_as_float(v[4 * u + 2]) * alpha, __uint_as_float(v[4 * u + 3]) * alpha);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
          if (threadIdx.x == 0 && m0 < M) {
#pragma unroll
            for (int j = 0; j < 2; ++j)
              if (n0 + 64 * q + 32 * j < N)
                asm volatile(
                    "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(&tmap_y),
                    "r"((int)(n0 + 64 * q + 32 * j)), "r"((int)m0), "r"(smem_addr(sm.ystage + j * (BM * 128)))
                    : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < 8; c += 2) {  // two loads in flight per wait
          uint32_t v0[32], v1[32];
          tmem_ld_32x32b_x32(acc + 32 * c, v0);
          tmem_ld_32x32b_x32(acc + 32 * c + 32, v1);
          tmem_wait_ld();
          if (row < M && n0 + 32 * c < N) store_row32<kF32>(y, row * N, n0 + 32 * c, N, v0, alpha, vec_ok);
          if (row < M && n0 + 32 * c + 32 < N) store_row32<kF32>(y, row * N, n0 + 32 * c + 32, N, v1, alpha, vec_ok);
        }
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(&sm.acc_free[b], lead);
      }
    }
    if (failed && lane == 0) atomicOr(status, kStatusTimeout);
    if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }
  // neither CTA leaves (or frees TMEM) while the other may still touch its
  // shared memory or TMEM
  fence_before_sync();
  __syncthreads();
  cluster_sync();
  if (warp == 0) {
    fence_after_sync();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Row-major [rows, row_bytes] uint8 matrix, boxes of [box_rows, 128 bytes],
// 128-byte swizzle, zero fill outside the matrix.
bool make_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_bytes, uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {row_bytes, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major [rows, pitch_bytes] matrix of which the first row_bytes of each
// row are the tensor (zero fill beyond them and past the last row), boxes of
// [128 rows, 128 bytes], 128-byte swizzle.
bool make_map_pitch(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_bytes, uint64_t pitch_bytes) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {row_bytes, rows};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {128, 128};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Y as bf16 [M, N] for TMA stores: boxes of 128 rows x 64 columns (128
// bytes), 128-byte swizzle.
// The output map for TMA stores: boxes of 128 rows x 128 bytes (64 bf16 or
// 32 fp32), 128-byte swizzle.  Rows of Y must be 16-byte aligned.
bool make_y_map(CUtensorMap* map, void* y, uint64_t M, uint64_t N, bool f32 = false) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {N, M};
  cuuint64_t strides[1] = {N * (f32 ? 4 : 2)};
  cuuint32_t box[2] = {f32 ? 32u : 64u, (cuuint32_t)BM};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, y, dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN>
cudaError_t launch_bn(const uint8_t* a_codes, const uint8_t* a_smma, const float* a_ts, int64_t M,
                      const uint8_t* w_codes, const uint8_t* w_smma, const float* w_ts, int64_t N, int64_t K,
                      void* y, bool out_f32, unsigned int* status, int num_sms, cudaStream_t stream) {
  CUtensorMap ma, mb, my;
  if (!make_map(&ma, a_codes, (uint64_t)M, (uint64_t)K / 2, BM) ||
      !make_map(&mb, w_codes, (uint64_t)N, (uint64_t)K / 2, BN))
    return cudaErrorInvalidValue;
  // TMA stores of the output: bf16, wide tiles, rows of Y 16-byte aligned
  int tma_store = (!out_f32 && BN == 256 && N % 8 == 0) ? 1 : 0;
  memset(&my, 0, sizeof my);
  if (tma_store && !make_y_map(&my, y, (uint64_t)M, (uint64_t)N)) tma_store = 0;
  // one CTA per SM: each allocates all 512 TMEM columns, which the block
  // scheduler does not count, so ask for enough shared memory that a second
  // CTA never lands on the same SM (228 KB per SM)
  const size_t smem = std::max<size_t>(sizeof(Smem<BN>) + 1024, 120u * 1024u);
  auto kern = out_f32 ? w4a4_kernel<BN, true> : w4a4_kernel<BN, false>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int64_t work = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::min<int64_t>(work, num_sms));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, ma, mb, my, tma_store, a_smma, w_smma, a_ts, w_ts, M, N, K, y, status);
}

std::atomic<int> g_cluster_ctas{2};

// Pair-kernel launch: clusters of 2 CTAs, one CTA per SM (the shared-memory
// request is above half an SM's), as many clusters as fit at once or as there
// are work units.  cudaErrorNotSupported when no pair can be resident.
template <bool kGateUp = false>
cudaError_t launch_pairs(const uint8_t* a_codes, const uint8_t* a_smma, const float* a_ts, int64_t M,
                         const uint8_t* w_codes, const uint8_t* w_smma, const float* w_ts, int64_t N, int64_t K,
                         void* y, bool out_f32, unsigned int* status, cudaStream_t stream) {
  CUtensorMap ma, mb, my;
  if (!make_map(&ma, a_codes, (uint64_t)M, (uint64_t)K / 2, 128) ||
      !make_map(&mb, w_codes, (uint64_t)N, (uint64_t)K / 2, 128))
    return cudaErrorInvalidValue;
  const int64_t n_out = kGateUp ? N / 2 : N;  // columns of Y
  // TMA stores of the output: rows of Y 16-byte aligned (fp32 as well, except
  // for the gate/up epilogue, which writes bf16 only)
  int tma_store = (out_f32 ? (!kGateUp && n_out % 4 == 0) : n_out % 8 == 0) ? 1 : 0;
  memset(&my, 0, sizeof my);
  if (tma_store && !make_y_map(&my, y, (uint64_t)M, (uint64_t)n_out, out_f32)) tma_store = 0;
  if (kGateUp && !tma_store) return cudaErrorNotSupported;
  const size_t smem = sizeof(PairSmem) + 1024;
  auto kern = out_f32 ? w4a4_pair_kernel<true> : w4a4_pair_kernel<false>;
  if constexpr (kGateUp) kern = w4a4_pair_kernel<false, true>;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kPairThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // resident clusters per GPU, once per output type (the device is fixed for the process)
  static int max_clusters[2] = {0, 0};  // per instantiation: [output f32]
  static std::once_flag once[2];
  cudaError_t err = cudaSuccess;
  std::call_once(once[out_f32 ? 1 : 0], [&] {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return;
    cudaLaunchConfig_t q = cfg;
    q.gridDim = dim3(2);
    q.numAttrs = 1;  // the cluster shape only
    int n = 0;
    err = cudaOccupancyMaxActiveClusters(&n, kern, &q);
    max_clusters[out_f32 ? 1 : 0] = err == cudaSuccess ? n : 0;
  });
  if (err != cudaSuccess) return err;
  const int mc = max_clusters[out_f32 ? 1 : 0];
  if (mc < 1) return cudaErrorNotSupported;
  const int64_t tiles_n = kGateUp ? N / 2 / 128 : (N + 255) / 256;
  const int64_t work = ((M + 255) / 256) * tiles_n;
  cfg.gridDim = dim3((unsigned)(2 * std::min<int64_t>(work, mc)));
  return cudaLaunchKernelEx(&cfg, kern, ma, mb, my, tma_store, a_smma, w_smma, a_ts, w_ts, M, N, K, y, status);
}

}  // namespace

cudaError_t launch_gemm_bf16_tn(const void* a, int64_t pitch_a, const void* b, int64_t pitch_b, int64_t rows_a,
                                int64_t rows_b, int64_t red, void* y, bool out_f32, unsigned int* status,
                                cudaStream_t stream) {
  if (rows_a <= 0 || rows_b <= 0) return cudaSuccess;
  if (red <= 0 || pitch_a < red || pitch_b < red || pitch_a % 8 != 0 || pitch_b % 8 != 0 || rows_a > INT32_MAX ||
      rows_b > INT32_MAX || red > ((int64_t)1 << 28))
    return cudaErrorNotSupported;
  CUtensorMap ma, mb, my;
  if (!make_map_pitch(&ma, a, (uint64_t)rows_a, (uint64_t)red * 2, (uint64_t)pitch_a * 2) ||
      !make_map_pitch(&mb, b, (uint64_t)rows_b, (uint64_t)red * 2, (uint64_t)pitch_b * 2))
    return cudaErrorInvalidValue;
  int tma_store = (out_f32 ? rows_b % 4 == 0 : rows_b % 8 == 0) ? 1 : 0;
  memset(&my, 0, sizeof my);
  if (tma_store && !make_y_map(&my, y, (uint64_t)rows_a, (uint64_t)rows_b, out_f32)) tma_store = 0;
  const size_t smem = sizeof(PairSmem) + 1024;
  auto kern = out_f32 ? w4a4_pair_kernel<true, false, true> : w4a4_pair_kernel<false, false, true>;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kPairThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  static int max_clusters[2] = {0, 0};  // per output type (the device is fixed for the process)
  static std::once_flag once[2];
  cudaError_t err = cudaSuccess;
  std::call_once(once[out_f32 ? 1 : 0], [&] {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return;
    cudaLaunchConfig_t q = cfg;
    q.gridDim = dim3(2);
    q.numAttrs = 1;  // the cluster shape only
    int n = 0;
    err = cudaOccupancyMaxActiveClusters(&n, kern, &q);
    max_clusters[out_f32 ? 1 : 0] = err == cudaSuccess ? n : 0;
  });
  if (err != cudaSuccess) return err;
  const int mc = max_clusters[out_f32 ? 1 : 0];
  if (mc < 1) return cudaErrorNotSupported;
  const int64_t work = ((rows_a + 255) / 256) * ((rows_b + 255) / 256);
  cfg.gridDim = dim3((unsigned)(2 * std::min<int64_t>(work, mc)));
  const int64_t k4 = 4 * ((red + 15) / 16 * 16);  // 16-wide MMA steps, counted as in the NVFP4 mode
  const uint8_t* no_sf = nullptr;
  const float* no_ts = nullptr;
  return cudaLaunchKernelEx(&cfg, kern, ma, mb, my, tma_store, no_sf, no_sf, no_ts, no_ts, rows_a, rows_b, k4, y,
                            status);
}

cudaError_t launch_gemm_w4a4_gate_up(const uint8_t* a_codes, const uint8_t* a_scales_mma, const float* a_ts,
                                     int64_t M, const uint8_t* w_codes, const uint8_t* w_scales_mma,
                                     const float* w_ts, int64_t N, int64_t K, void* y, unsigned int* status,
                                     int num_sms, cudaStream_t stream) {
  if (M <= 0) return cudaSuccess;
  if (N % 256 != 0 || K < BK || K % 64 != 0 || M > INT32_MAX || N > INT32_MAX) return cudaErrorNotSupported;
  if (M > BM && w4a4_get_cluster_ctas() >= 2)
    return launch_pairs<true>(a_codes, a_scales_mma, a_ts, M, w_codes, w_scales_mma, w_ts, N, K, y, false, status,
                              stream);
  // single CTAs, one per 128-feature tile (256 weight rows: gate, then up)
  const int64_t F = N / 2;
  CUtensorMap ma, mb, my;
  if (!make_map(&ma, a_codes, (uint64_t)M, (uint64_t)K / 2, BM) ||
      !make_map(&mb, w_codes, (uint64_t)N, (uint64_t)K / 2, 128))
    return cudaErrorInvalidValue;
  memset(&my, 0, sizeof my);
  if (!make_y_map(&my, y, (uint64_t)M, (uint64_t)F)) return cudaErrorNotSupported;
  const size_t smem = std::max<size_t>(sizeof(Smem<256>) + 1024, 120u * 1024u);  // one CTA per SM (see launch_bn)
  auto kern = w4a4_kernel<256, false, true>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int64_t work = ((M + BM - 1) / BM) * (F / 128);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::min<int64_t>(work, num_sms));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, ma, mb, my, 1, a_scales_mma, w_scales_mma, a_ts, w_ts, M, N, K, y, status);
}

bool w4a4_set_cluster_ctas(int ctas) {
  if (ctas != 1 && ctas != 2) return false;
  g_cluster_ctas.store(ctas, std::memory_order_relaxed);
  return true;
}
int w4a4_get_cluster_ctas() { return g_cluster_ctas.load(std::memory_order_relaxed); }

cudaError_t launch_gemm_w4a4(const uint8_t* a_codes, const uint8_t* a_scales_mma, const float* a_ts, int64_t M,
                             const uint8_t* w_codes, const uint8_t* w_scales_mma, const float* w_ts, int64_t N,
                             int64_t K, void* y, bool out_f32, unsigned int* status, int num_sms,
                             cudaStream_t stream) {
  if (M <= 0) return cudaSuccess;
  if (K < BK || K % 64 != 0 || M > INT32_MAX || N > INT32_MAX) return cudaErrorNotSupported;
  if (M <= BM) {
    // one CTA per weight tile, the narrowest tile (64, 128 or 256 rows) whose
    // tiles fit one wave: each CTA streams one tile's rows
    if ((N + 63) / 64 <= num_sms)
      return launch_bn<64>(a_codes, a_scales_mma, a_ts, M, w_codes, w_scales_mma, w_ts, N, K, y, out_f32, status,
                           num_sms, stream);
    if ((N + 127) / 128 <= num_sms)
      return launch_bn<128>(a_codes, a_scales_mma, a_ts, M, w_codes, w_scales_mma, w_ts, N, K, y, out_f32, status,
                            num_sms, stream);
    return launch_bn<256>(a_codes, a_scales_mma, a_ts, M, w_codes, w_scales_mma, w_ts, N, K, y, out_f32, status,
                          num_sms, stream);
  }
  const int ctas = w4a4_get_cluster_ctas();
  cudaError_t err = cudaErrorNotSupported;
  if (ctas == 2)
    err = launch_pairs<false>(a_codes, a_scales_mma, a_ts, M, w_codes, w_scales_mma, w_ts, N, K, y, out_f32, status,
                          stream);
  if (err != cudaErrorNotSupported) return err;
  return launch_bn<256>(a_codes, a_scales_mma, a_ts, M, w_codes, w_scales_mma, w_ts, N, K, y, out_f32, status,
                        num_sms, stream);
}

}  // namespace nvfp4
