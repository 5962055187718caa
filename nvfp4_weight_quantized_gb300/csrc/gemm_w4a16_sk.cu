// gemm_w4a16_sk.cu -- decode-sized W4A16 (bf16 activations x NVFP4 weights,
// fp32 accumulation): persistent split-K with the activations resident in
// shared memory as f16.
//
// The small-M path of "SOAR 2026 Recap ...", section "1. Quantization and
// GEMM dispatch" (W4A16 below the crossover).  At M <= 64 tokens the GEMM is
// a weight stream (0.5625 bytes of codes and scales per weight), and one SM
// must dequantise its share of the HBM stream (~20 bytes per SM cycle), so
// the kernel keeps the per-byte instruction count minimal:
//
// Work division.  One CTA per SM, in clusters of ks <= 8 CTAs.  CTA rank r of
// a cluster owns K slice r (a run of 256-wide stages) of every 128-row tile
// its cluster handles (tiles c, c + G, ... for cluster c of G).  Every CTA
// keeps the partial tile of each of its tiles in shared memory; after the
// last one a single cluster barrier, then each CTA sums 128 / ks of the rows
// of every tile over the ks slices through distributed shared memory and
// stores them -- no synchronisation between CTAs while the weights stream.
// A producer warp streams the weight codes (TMA, 128 x 128-byte boxes,
// 128-byte swizzle) and MMA-tiled scales (bulk copies) of every (tile,
// stage) through a ring, continuously across tiles.
//
// Arithmetic.
//   * X: at the start every CTA loads its K slice of the activations once,
//     finds each token's largest magnitude there and stores the slice in
//     shared memory as f16 times the power of two that puts that maximum into
//     [2^15, 65280] -- exact for every element within 2^29 of it (smaller ones
//     round to f16 subnormals, far below the fp32 accumulation error);
//   * W: the hardware E2M1x2 -> f16x2 conversion gives the two weights of a
//     code byte exactly and one f16x2 multiply by the E4M3 block scale (also
//     exact in f16) gives value * scale (at most 6 significant bits, within
//     [2^-10, 2688]): two instructions per code byte;
//   * m16n8k16 f16 MMAs, fp32 accumulation.  Warp w owns 16 weight rows;
//     thread (g, t) dequantises rows g and g+8, K positions [16t, 16t+16) of
//     a 64-wide chunk -- one 16-element scale block -- so the operand layout
//     is met by permuting which K positions each MMA step sees (the same
//     permutation for the weights and for X, so the sum is unchanged): step j
//     takes code bytes 8t+2j and 8t+2j+1, i.e. K = 16t+4j .. 16t+4j+3;
//   * a partial tile leaves in real units: times ts, then times 2^(e - 142)
//     for each token, so no intermediate overflows or underflows unless the
//     result does.
// Every mbarrier wait is bounded; launched with programmatic dependent launch
// (set-up and, for static weights, the first weight copies overlap the
// previous kernel; X is read after the wait).
#include <cuda.h>
#include <cuda_bf16.h>

#include <map>
#include <mutex>
#include <tuple>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"
#include "w4a16_frag.cuh"

namespace nvfp4 {

namespace {

using namespace sm100;
using namespace w4a16;

constexpr int BM = 128;                 // weight rows per tile
constexpr int kChunkK = 64;             // K per MMA group (4 steps of 16)
constexpr int kStageK = 256;            // K per pipeline stage
constexpr int kChunksPerStage = kStageK / kChunkK;
constexpr int kRowWarps = 8;            // 16 rows each
constexpr int kCodeBytes = BM * kStageK / 2;                 // 16 KB per stage
constexpr int kSfBytes = kChunksPerStage * kScaleTileBytes;  // 2 KB per stage
constexpr int kMaxTok = 64;
constexpr int kMaxCluster = 8;
constexpr int kMaxStages = 8;
constexpr int kRedStride = BM + 4;      // fp32 words per token row of a partial tile
constexpr int kExpFloor = 16;           // token exponents are taken at least this large
constexpr uint32_t kSmemBudget = 220u * 1024u;

// Compute warps: kRowWarps * SPLIT, SPLIT warps per row group taking the
// chunks of a stage in turn (2 for narrow token tiles, where more warps hide
// more latency; 1 for wide ones, whose accumulators need the registers); the
// producer warp comes last.
constexpr int split_for(int nt) { return nt <= 2 ? 2 : 1; }
template <int SPLIT>
struct Warps {
  static constexpr int kCompute = kRowWarps * SPLIT;
  static constexpr int kProducer = kCompute;
  static constexpr int kThreads = 32 * (kCompute + 1);
};

struct Layout {
  uint32_t x_tile, x_off, codes_off, sf_off, pb_off, tok_off, bar_off, total;
  __host__ __device__ Layout(int st, int nt, int sps, int tiles) {
    x_tile = (uint32_t)nt * 128u;                        // one 64-wide chunk: token rows of 128 bytes
    x_off = 0;                                           // the resident K slice: 4 * sps chunks
    codes_off = ((uint32_t)sps * kChunksPerStage * x_tile + 1023u) & ~1023u;
    sf_off = codes_off + (uint32_t)st * kCodeBytes;
    pb_off = sf_off + (uint32_t)st * kSfBytes;           // partial tiles [tiles][nt][kRedStride] fp32
    tok_off = pb_off + (uint32_t)(tiles > 1 ? tiles : 1) * nt * kRedStride * 4u;  // per token: max |x| bits, then e
    bar_off = (tok_off + (uint32_t)nt * 4u + 7u) & ~7u;
    total = bar_off + 2u * kMaxStages * 8u + 1024u;      // + alignment slack
  }
};

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

__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t local_saddr, uint32_t rank) {
  uint32_t remote;
  asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_saddr), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(remote));
  return v;
}

template <int NT, bool kF32, int SPLIT = split_for(NT), typename Wp = Warps<SPLIT>>
__global__ void __launch_bounds__(Wp::kThreads, 1)
w4a16_sk_kernel(const __grid_constant__ CUtensorMap tmap_codes, const __nv_bfloat16* __restrict__ x,
                const uint8_t* __restrict__ smma, const float* __restrict__ ts_ptr, int64_t M, int64_t N,
                int64_t K, int stages, int sps, int tiles_n, int clusters, int log2_ks, int max_tiles, int prefetch_w,
                void* __restrict__ y, unsigned int* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int n_tok = 8 * NT;
  constexpr int kComputeWarps = Wp::kCompute, kProducerWarp = Wp::kProducer, kThreads = Wp::kThreads;
  const Layout L(stages, n_tok, sps, max_tiles);
  uint64_t* full = reinterpret_cast<uint64_t*>(base + L.bar_off);
  uint64_t* empty = full + kMaxStages;
  uint32_t* tmax = reinterpret_cast<uint32_t*>(base + L.tok_off);
  const uint32_t sbase = smem_addr(base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int ks = 1 << log2_ks;
  const int cid = (int)(blockIdx.x >> log2_ks);
  const int rank = (int)cluster_ctarank();
  const int nchunk = (int)(K / kChunkK);
  const int nstage = (nchunk + kChunksPerStage - 1) / kChunksPerStage;
  const int st_begin = rank * sps;
  const int nst = max(0, min(st_begin + sps, nstage) - st_begin);  // this CTA's stages per tile
  const int ntiles = cid < tiles_n ? (tiles_n - 1 - cid) / clusters + 1 : 0;
  const int nunits = ntiles * nst;
  const int64_t ct = K / 64;

  if (threadIdx.x == kProducerWarp * 32) {
    prefetch_tmap(&tmap_codes);
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kComputeWarps);
    }
    fence_mbar_init();
  }
  if (threadIdx.x < n_tok) tmax[threadIdx.x] = 0u;
  __syncthreads();

  auto chunks_at = [&](int st) { return min(kChunksPerStage, nchunk - kChunksPerStage * st); };
  // unit i = (tile cid + (i / nst) * clusters, stage st_begin + i % nst), tracked
  // incrementally (no divisions)
  auto issue_w = [&](int s, int tile, int st) {
    const int ch = chunks_at(st);
    mbar_arrive_expect_tx(&full[s], (uint32_t)(kCodeBytes + ch * kScaleTileBytes));
    tma_load_2d(base + L.codes_off + s * kCodeBytes, &tmap_codes, st * (kStageK / 2), tile * BM, &full[s]);
    bulk_load(base + L.sf_off + s * kSfBytes, smma + ((int64_t)tile * ct + (int64_t)kChunksPerStage * st) * kScaleTileBytes,
              (uint32_t)ch * kScaleTileBytes, &full[s]);
  };
  const bool producer = threadIdx.x == kProducerWarp * 32;
  const int first = min(nunits, stages);
  int p_tile = cid, p_st = st_begin;  // producer position after the initial fill
  auto p_next = [&]() {
    if (++p_st == st_begin + nst) {
      p_st = st_begin;
      p_tile += clusters;
    }
  };
  // Weights declared static (nvfp4_set_weight_prefetch) are requested before
  // the wait on the previous kernel, overlapping its epilogue.
  if (producer && prefetch_w)
    for (int i = 0; i < first; ++i, p_next()) issue_w(i, p_tile, p_st);
  griddep_wait();  // X and ts (and possibly W) come from earlier kernels; Y may be read by them
  if (producer && !prefetch_w)
    for (int i = 0; i < first; ++i, p_next()) issue_w(i, p_tile, p_st);

  // ---- the resident X slice: per-token maxima, then f16 * 2^(142 - e) ----
  const int64_t k0 = (int64_t)st_begin * kStageK;
  const int kl = (int)(min(K, k0 + (int64_t)nst * kStageK) - k0);  // K of this slice (multiple of 64)
  const int upt = kl / 8;                                           // 16-byte pieces per token row
  const int m_valid = (int)(M < n_tok ? M : (int64_t)n_tok);
  // thread i works on token i / kTpt (kTpt threads per token), pieces
  // i % kTpt + j * kTpt, four loads in flight; partial maxima go to 8 slots
  // per token, then one slot holds the token's maximum
  constexpr int kTpt = kThreads / n_tok;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(base + L.pb_off);  // [n_tok][8], before the partial tiles
  for (int i = threadIdx.x; i < n_tok * 8; i += kThreads) tslot[i] = 0u;
  __syncthreads();
  const int my_tok = threadIdx.x / kTpt, my_sub = threadIdx.x - my_tok * kTpt;
  const bool has_tok = my_tok < n_tok, loads = my_tok < m_valid;
  const uint4* my_row = reinterpret_cast<const uint4*>(x + (int64_t)(loads ? my_tok : 0) * K + k0);
  // up to kHold pieces per thread are read once and kept in registers; a
  // longer slice is read twice
  constexpr int kHold = 8;
  const bool hold = upt <= kHold * kTpt;
  uint4 hv[kHold];
  if (has_tok && loads) {
    uint32_t mx = 0;
    if (hold) {
#pragma unroll
      for (int j = 0; j < kHold; ++j) {
        const int u = my_sub + j * kTpt;
        hv[j] = u < upt ? __ldg(my_row + u) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int j = 0; j < kHold; ++j)
        mx = max_u16x2(mx, max_u16x2(max_u16x2(hv[j].x & 0x7FFF7FFFu, hv[j].y & 0x7FFF7FFFu),
                                     max_u16x2(hv[j].z & 0x7FFF7FFFu, hv[j].w & 0x7FFF7FFFu)));
    } else {
      for (int u = my_sub; u < upt; u += 4 * kTpt) {
        uint4 v[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) v[r] = u + r * kTpt < upt ? __ldg(my_row + u + r * kTpt) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int r = 0; r < 4; ++r)
          mx = max_u16x2(mx, max_u16x2(max_u16x2(v[r].x & 0x7FFF7FFFu, v[r].y & 0x7FFF7FFFu),
                                       max_u16x2(v[r].z & 0x7FFF7FFFu, v[r].w & 0x7FFF7FFFu)));
      }
    }
    mx = max(mx & 0xFFFFu, mx >> 16);
    if (mx != 0u) atomicMax(&tslot[my_tok * 8 + (my_sub & 7)], mx);
  }
  __syncthreads();
  if (threadIdx.x < n_tok) {
    uint32_t mx = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) mx = max(mx, tslot[threadIdx.x * 8 + j]);
    tmax[threadIdx.x] = (uint32_t)max(kExpFloor, (int)(mx >> 7));
  }
  __syncthreads();
  // chunk q of the slice: token row r at r * 128, 16-byte unit u at u ^ (r & 7)
  if (has_tok) {
    const float c = exp2i(142 - (int)tmax[my_tok]);
    const uint32_t xrow = sbase + L.x_off + my_tok * 128;
    auto put = [&](int u, uint4 v) {
      sts128(xrow + (u >> 3) * L.x_tile + (((u & 7) ^ (my_tok & 7)) << 4),
             make_uint4(bf16x2_to_f16x2(v.x, c), bf16x2_to_f16x2(v.y, c), bf16x2_to_f16x2(v.z, c),
                        bf16x2_to_f16x2(v.w, c)));
    };
    if (hold) {
#pragma unroll
      for (int j = 0; j < kHold; ++j) {
        const int u = my_sub + j * kTpt;
        if (u < upt) put(u, loads ? hv[j] : make_uint4(0, 0, 0, 0));
      }
    } else {
      for (int u = my_sub; u < upt; u += 4 * kTpt) {
        uint4 v[4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
          v[r] = (loads && u + r * kTpt < upt) ? __ldg(my_row + u + r * kTpt) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int r = 0; r < 4; ++r)
          if (u + r * kTpt < upt) put(u + r * kTpt, v[r]);
      }
    }
  }
  __syncthreads();

  bool failed = false;
  if (warp == kProducerWarp) {
    if (lane == 0) {
      int s = 0;
      uint32_t eph = 0;  // units past the first `stages` reuse slots in order
      for (int i = first; i < nunits; ++i, p_next()) {
        if (!mbar_wait(&empty[s], eph)) {
          failed = true;
          break;
        }
        issue_w(s, p_tile, p_st);
        if (++s == stages) {
          s = 0;
          eph ^= 1u;
        }
      }
      if (failed) atomicOr(status, kStatusTimeout);
    }
  } else {
    // After a wait runs out, `failed` is set and later waits are skipped,
    // but every loop keeps its trip count, so the compute warps still meet at
    // every named barrier and the CTA reaches the final cluster barrier.
    const float tsv = *ts_ptr;
    const int g = lane >> 2, t = lane & 3;
    const int r0 = (warp % kRowWarps) * 16 + g, r1 = r0 + 8;
    const int par = warp / kRowWarps;  // this warp takes the chunks q of a stage with q % SPLIT == par
    // code rows: 128 bytes each, 16-byte unit u stored at u ^ (row & 7); both
    // rows of this thread have (row & 7) == g.  Chunk q, thread t reads bytes
    // 32q + 8t .. +8: unit 2q + t/2, half t & 1.
    const uint32_t crow0 = (uint32_t)(r0 * 128 + (t & 1) * 8), crow1 = (uint32_t)(r1 * 128 + (t & 1) * 8);
    const uint32_t sf0 = (uint32_t)((r0 & 31) * 16 + (r0 >> 5) * 4 + t);
    const uint32_t sf1 = (uint32_t)((r1 & 31) * 16 + (r1 >> 5) * 4 + t);
    uint32_t xoff[NT][2];
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      const int tok = 8 * i + g;
      xoff[i][0] = (uint32_t)(tok * 128 + (((2 * t) ^ (tok & 7)) << 4));
      xoff[i][1] = (uint32_t)(tok * 128 + (((2 * t + 1) ^ (tok & 7)) << 4));
    }
    // real-unit factors of this thread's accumulator columns (tokens 8n+2t, 8n+2t+1)
    float u0[NT], u1[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      u0[n] = exp2i((int)tmax[8 * n + 2 * t] - 142);
      u1[n] = exp2i((int)tmax[8 * n + 2 * t + 1] - 142);
    }
    int s = 0;
    uint32_t ph = 0;
    for (int it = 0; it < ntiles; ++it) {
      float acc[NT][4];
      float acc2[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // second chain for a single token tile
#pragma unroll
      for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.0f;
      for (int sl = 0; sl < nst; ++sl) {
        if (!failed && !mbar_wait(&full[s], ph)) failed = true;
        const int chunks = chunks_at(st_begin + sl);
        const uint32_t cb = sbase + L.codes_off + s * kCodeBytes;
        const uint32_t sb = sbase + L.sf_off + s * kSfBytes;
        const uint32_t xs = sbase + L.x_off + (uint32_t)(sl * kChunksPerStage) * L.x_tile;
        auto chunk = [&](int q) {
          const uint32_t unit = (uint32_t)((((2 * q + (t >> 1)) ^ g)) << 4);
          const uint2 w0 = lds64(cb + crow0 + unit), w1 = lds64(cb + crow1 + unit);
          const uint32_t s0 = scale_f16x2(lds8(sb + q * kScaleTileBytes + sf0));
          const uint32_t s1 = scale_f16x2(lds8(sb + q * kScaleTileBytes + sf1));
          uint32_t a0[8], a1[8];  // f16x2 of bytes 8t .. 8t+7 of rows r0 and r1
          dequant4(w0.x, s0, a0);
          dequant4(w0.y, s0, a0 + 4);
          dequant4(w1.x, s1, a1);
          dequant4(w1.y, s1, a1 + 4);
          const uint32_t xb = xs + q * L.x_tile;
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
        };
        if (chunks == kChunksPerStage) {  // full stage: unrolled, so the chunks overlap
#pragma unroll
          for (int k = 0; k < kChunksPerStage / SPLIT; ++k) chunk(par + k * SPLIT);
        } else {
          for (int q = par; q < chunks; q += SPLIT) chunk(q);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_cta(&empty[s]);
        if (++s == stages) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (NT == 1) {
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[0][e] += acc2[e];
      }

      // ---- the tile's partial (this K slice) -> slot it, in real units ----
      float* pb = reinterpret_cast<float*>(base + L.pb_off) + it * n_tok * kRedStride;
      for (int phs = SPLIT - 1; phs >= 0; --phs) {
        if (par == phs) {
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            float* p0 = pb + (8 * n + 2 * t) * kRedStride + r0;
            float* p1 = p0 + kRedStride;
            const float v0 = (acc[n][0] * tsv) * u0[n], v1 = (acc[n][1] * tsv) * u1[n];
            const float v2 = (acc[n][2] * tsv) * u0[n], v3 = (acc[n][3] * tsv) * u1[n];
            if (phs == SPLIT - 1) {
              p0[0] = v0;
              p1[0] = v1;
              p0[8] = v2;
              p1[8] = v3;
            } else {
              p0[0] += v0;
              p1[0] += v1;
              p0[8] += v2;
              p1[8] += v3;
            }
          }
        }
        if (SPLIT > 1 && phs > 0) asm volatile("bar.sync 1, %0;" ::"n"(kComputeWarps * 32) : "memory");
      }
    }
    if (failed && lane == 0) atomicOr(status, kStatusTimeout);
  }
  __syncwarp();
  // The next kernel in the stream may start its prologue now (it waits for
  // this grid to finish before it touches data).
  griddep_launch_dependents();
  cluster_sync_all();  // every partial tile of the cluster is in (and every peer is running)
  // ---- rows [rank * 128 / ks, (rank + 1) * 128 / ks) of every tile: the ks
  // slices summed in rank order, stored ----
  {
    const int rows = BM / ks, rlo = rank * rows, per_tok = rows / 4;
    const int per_tile = m_valid * per_tok;
    for (int i = threadIdx.x; i < ntiles * per_tile; i += kThreads) {
      const int it = i / per_tile, j = i - it * per_tile;
      const int tk = j / per_tok, row = rlo + 4 * (j - tk * per_tok);
      const uint32_t a = sbase + L.pb_off + (uint32_t)((it * n_tok + tk) * kRedStride + row) * 4u;
      float4 v[kMaxCluster];
#pragma unroll
      for (int q = 0; q < kMaxCluster; ++q)
        if (q < ks) v[q] = ld_dsmem_f4(a, (uint32_t)q);
      float4 sum = v[0];
#pragma unroll
      for (int q = 1; q < kMaxCluster; ++q)
        if (q < ks) {
          sum.x += v[q].x;
          sum.y += v[q].y;
          sum.z += v[q].z;
          sum.w += v[q].w;
        }
      const int64_t n = (int64_t)(cid + it * clusters) * BM + row;
      const float o[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (n + e < N) {
          if (kF32) static_cast<float*>(y)[tk * N + n + e] = o[e];
          else static_cast<__nv_bfloat16*>(y)[tk * N + n + e] = __float2bfloat16_rn(o[e]);
        }
      }
    }
  }
  // peers may still read this CTA's partial tiles: leave together
  __syncwarp();
  cluster_sync_all();
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

bool make_codes_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_bytes) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {row_bytes, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {kStageK / 2, BM};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NT>
void* kernel_for(bool f32, int* threads) {
  *threads = Warps<split_for(NT)>::kThreads;
  return f32 ? (void*)w4a16_sk_kernel<NT, true> : (void*)w4a16_sk_kernel<NT, false>;
}

}  // namespace

// The largest M the resident-activation kernel takes.
int w4a16_sk_max_tokens() { return kMaxTok; }

cudaError_t launch_gemm_w4a16_sk(const void* x, int64_t M, const uint8_t* codes, const uint8_t* scales_mma,
                                 const float* ts, int64_t N, int64_t K, void* y, bool out_f32, bool prefetch_w,
                                 unsigned int* status, int num_sms, cudaStream_t stream) {
  if (M <= 0) return cudaSuccess;
  if (M > kMaxTok || K % 64 != 0 || N > INT32_MAX || K > INT32_MAX / 2) return cudaErrorNotSupported;
  int NT = (int)((M + 7) / 8);
  if (NT == 5) NT = 6;
  if (NT == 7) NT = 8;
  const int n_tok = 8 * NT;
  const int64_t tiles_n = (N + BM - 1) / BM;
  if (tiles_n > INT32_MAX / 2) return cudaErrorNotSupported;
  const int nstage = (int)((K / kChunkK + kChunksPerStage - 1) / kChunksPerStage);
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

  // Choose the cluster size ks (K slices) and the ring depth: the shared
  // memory must hold the f16 activation slice, two partial tiles and at least
  // two stages; among those, the fewest stage units per CTA (tiles per
  // cluster times stages per slice, plus two per tile for the sum).
  static std::mutex mu;
  static std::map<std::tuple<void*, int, uint32_t>, int> occ;  // (kernel, ks, smem) -> clusters at once
  int best_ks = 0, best_sps = 0, best_st = 0, best_cl = 0;
  int64_t best_cost = INT64_MAX;
  for (int ks = 1; ks <= kMaxCluster; ks *= 2) {
    const int sps = (nstage + ks - 1) / ks;
    if ((nstage + sps - 1) / sps != ks) continue;  // every rank gets stages
    // the partial tiles of all a cluster's tiles stay in shared memory: size
    // for the tiles per cluster at the cluster count that fits, found by
    // asking the occupancy calculator for the shared memory it implies
    int per = (int)((tiles_n + std::max(1, num_sms / ks) - 1) / std::max(1, num_sms / ks));
    int st = 0, cl = 0;
    uint32_t smem = 0;
    for (int iter = 0; iter < 3; ++iter) {
      st = kMaxStages;
      while (st > 2 && Layout(st, n_tok, sps, per).total > kSmemBudget) --st;
      smem = Layout(st, n_tok, sps, per).total;
      if (smem > kSmemBudget) break;
      cudaLaunchConfig_t q = {};
      q.blockDim = dim3((unsigned)threads);
      q.dynamicSmemBytes = smem;
      q.gridDim = dim3((unsigned)(ks * num_sms));
      cudaLaunchAttribute a[1];
      a[0].id = cudaLaunchAttributeClusterDimension;
      a[0].val.clusterDim.x = (unsigned)ks;
      a[0].val.clusterDim.y = 1;
      a[0].val.clusterDim.z = 1;
      q.attrs = a;
      q.numAttrs = 1;
      {
        std::lock_guard<std::mutex> lk(mu);
        auto it = occ.find({kern, ks, smem});
        if (it != occ.end()) {
          cl = it->second;
        } else {
          if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
              cudaOccupancyMaxActiveClusters(&cl, kern, &q) != cudaSuccess)
            cl = 0;
          occ[{kern, ks, smem}] = cl;
        }
      }
      if (cl < 1) break;
      const int64_t used = std::min<int64_t>(cl, tiles_n);
      const int need = (int)((tiles_n + used - 1) / used);
      if (need <= per) {
        cl = (int)used;
        break;
      }
      per = need;
      cl = 0;
    }
    if (cl < 1 || smem > kSmemBudget) continue;
    const int64_t cost = (int64_t)((tiles_n + cl - 1) / cl) * sps;
    if (cost < best_cost) {
      best_cost = cost;
      best_ks = ks;
      best_sps = sps;
      best_st = st;
      best_cl = cl;
    }
  }
  if (best_ks == 0) return cudaErrorNotSupported;
  int stages = best_st;
  const int max_tiles = (int)((tiles_n + best_cl - 1) / best_cl);
  const int64_t units = (int64_t)max_tiles * best_sps;
  if (stages > units) stages = (int)std::max<int64_t>(1, units);
  const uint32_t smem = Layout(stages, n_tok, best_sps, max_tiles).total;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;

  CUtensorMap mc;
  if (!make_codes_map(&mc, codes, (uint64_t)N, (uint64_t)K / 2)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(best_cl * best_ks));
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)best_ks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  int pf = prefetch_w ? 1 : 0, tn = (int)tiles_n, sps = best_sps, cl = best_cl, mt = max_tiles;
  int lks = 0;
  while ((1 << lks) < best_ks) ++lks;
  void* args[] = {(void*)&mc, (void*)&x,      (void*)&scales_mma, (void*)&ts, (void*)&M,   (void*)&N,
                  (void*)&K,  (void*)&stages, (void*)&sps,        (void*)&tn, (void*)&cl,  (void*)&lks,
                  (void*)&mt, (void*)&pf,     (void*)&y,          (void*)&status};
  return cudaLaunchKernelExC(&cfg, kern, args);
}

}  // namespace nvfp4
