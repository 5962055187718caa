// gemm_w4a16.cu -- bf16 activations x NVFP4 weights on the 5th-generation
// tensor cores, fp32 accumulation in TMEM.
//
// The small-M path of "SOAR 2026 Recap ...", section "1. Quantization and
// GEMM dispatch" (W4A16 for M <= 48 on the pages' GPU).  Decode-sized GEMMs
// stream 0.5625 bytes per weight from HBM and need about 3.6 * M flop per byte
// of weights, so at M = 48 the contraction alone is ~1.2 PFLOP/s at the HBM
// rate -- beyond the legacy mma.sync path (~0.6 PFLOP/s bf16 on this part) but
// a fraction of tcgen05.  The kernel therefore:
//   * streams the weight codes of a 128-row x K-slice tile with TMA (128-byte
//     swizzle) and the matching MMA-tiled scales with bulk copies, several
//     stages in flight, together with the activation tile X[tokens, k] (TMA,
//     128-byte swizzle, the layout the MMA reads as its B operand);
//   * dequantises in registers, one weight row per thread: E2M1 bits are
//     placed into bf16 bit positions (value * 2^-126 exactly) and one bf16x2
//     multiply by value(scale) * 2^119 gives value * scale * 2^-7, exact in
//     bf16; the result goes to TMEM with tcgen05.st;
//   * issues tcgen05.mma kind::f16 with A (the dequantised weights, M = 128
//     rows) read from TMEM and B (tokens, N = 16..128) from shared memory,
//     accumulating Y^T in TMEM;
//   * splits K across a thread-block cluster of up to 8 CTAs and reduces the
//     fp32 partial tiles through distributed shared memory (fixed order, no
//     global scratch); 2^7 * ts is applied in the epilogue.
// Warps 0-7 dequantise (warps w and w+4 share TMEM lanes 32*(w%4).., taking
// alternate K chunks) and warps 0-3 run the epilogue (TMEM lanes 0-127 =
// weight rows); warp 8 issues the TMA copies, warp 9 the MMAs.  Launched with
// programmatic dependent launch: set-up overlaps the previous kernel, and
// inputs are read only after griddepcontrol.wait.  Every mbarrier wait is
// bounded.
#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace nvfp4 {

namespace {

using namespace sm100;

constexpr int BM = 128;              // weight rows per CTA = MMA M = TMEM lanes
constexpr int kStageK = 256;         // K per pipeline stage (128 code bytes per row)
constexpr int kChunkK = 64;          // K per dequant chunk (4 MMAs of K = 16)
constexpr int kMaxTok = 64;          // tokens per CTA = MMA N (multiple of 16)
constexpr int kASlots = 4;           // TMEM A buffers (one chunk each)
constexpr int kDqWarps = 8;          // two dequant warps per 32-lane TMEM quarter
// Two MMA-issuing warps: one tcgen05.mma stream is bound by its issuer's
// latency (~110 cycles per K=16 MMA with A in TMEM), and two streams into two
// accumulators overlap on the tensor core.  Warp kMmaWarp + p issues the
// chunks with c % 2 == p into accumulator p.
constexpr int kProducerWarp = kDqWarps, kMmaWarp = kDqWarps + 1;
constexpr int kThreads = 32 * (kDqWarps + 3);
constexpr uint32_t kTmemCols = 256;
// Two accumulators (even / odd K chunks) so consecutive MMAs do not wait on
// each other's accumulation; the epilogue adds them.
constexpr uint32_t kAccCol = 0;      // accumulator j at kAccCol + 64 * j, up to 64 fp32 columns each
constexpr uint32_t kACol = 128;      // 4 slots x 32 columns (64 bf16 per row)
static_assert(kACol + 32 * kASlots <= kTmemCols && kMaxTok <= 64, "TMEM layout");
constexpr int kMaxCluster = 8;
constexpr int kCodesBytes = BM * 128;   // per stage
constexpr int kSfBytes = 4 * kScaleTileBytes;
// Dynamic shared memory that keeps a third CTA off an SM (228 KB per SM, 1 KB
// reserved per CTA): 3 * (77 KB + 1 KB) > 228 KB.
constexpr uint32_t kSmemFor2PerSm = 77u * 1024u;

struct Barriers {
  uint64_t full[4];
  uint64_t empty[4];
  uint64_t a_full[kASlots];
  uint64_t a_free[kASlots];
  uint64_t acc[2];
  uint32_t tmem_base;
};

struct Layout {  // dynamic shared memory, offsets from a 1024-aligned base
  int stages, n_tok;
  uint32_t x_bytes;   // one 64-wide K sub-tile of X: n_tok rows x 128 bytes
  uint32_t stage_bytes, bar_off, total;
  __host__ __device__ Layout(int st, int nt) : stages(st), n_tok(nt) {
    x_bytes = (uint32_t)nt * 128u;
    stage_bytes = kCodesBytes + 4 * x_bytes + kSfBytes;  // all multiples of 1024
    bar_off = (uint32_t)st * stage_bytes;
    total = bar_off + (uint32_t)sizeof(Barriers) + 1024;
  }
  __device__ uint32_t codes(int s) const { return s * stage_bytes; }
  __device__ uint32_t x(int s, int q) const { return s * stage_bytes + kCodesBytes + q * x_bytes; }
  __device__ uint32_t sf(int s) const { return s * stage_bytes + kCodesBytes + 4 * x_bytes; }
};

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// value(E4M3 byte) * 2^119 as a bf16 pair (exact: at most 4 significant bits).
__device__ __forceinline__ uint32_t scale_pair(uint32_t sbyte) {
  const uint32_t sb = __float_as_uint(e4m3_to_f32(sbyte) * 0x1p119f) >> 16;
  return sb | (sb << 16);
}

// 4 code bytes (8 elements) -> 4 bf16x2 words value * scale * 2^-7; word i
// holds elements (2i, 2i+1) with the lower index in the low half.
__device__ __forceinline__ void dequant8(uint32_t v, uint32_t s2, uint32_t* out) {
  const uint32_t v4 = v >> 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    // low nibble of byte i -> bits 3:0, high nibble of byte i -> bits 19:16
    uint32_t z = __byte_perm(v, v4, (uint32_t)(i | (i << 4) | ((4 + i) << 8) | ((4 + i) << 12)));
    z &= 0x000F000Fu;
    // magnitude bits -> bf16 bits 8:6 (exponent 1:0, top mantissa bit), sign -> bit 15
    z = (z * 0x1040u) & 0x81C081C0u;
    out[i] = bf16x2_mul(z, s2);
  }
}

__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, bf16 inputs, fp32 accumulation, K = 16.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
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
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_saddr), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(remote)
               : "memory");
  return v;
}

template <bool kF32>
__device__ __forceinline__ void store_out(void* y, int64_t idx, float v) {
  if (kF32) static_cast<float*>(y)[idx] = v;
  else static_cast<__nv_bfloat16*>(y)[idx] = __float2bfloat16_rn(v);
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), A and
// B bf16 (bits 7-9 and 10-12 = 1), both K-major, N >> 3 in bits 17-22,
// M >> 4 in bits 24-28.
__device__ __forceinline__ uint32_t idesc_bf16(int n_tok) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n_tok >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

template <bool kF32>
__global__ void __launch_bounds__(kThreads, 1)
w4a16_tc_kernel(const __grid_constant__ CUtensorMap tmap_codes, const __grid_constant__ CUtensorMap tmap_x,
                const uint8_t* __restrict__ smma, const float* __restrict__ ts_ptr, int64_t M, int64_t N,
                int64_t K, int n_tok, int stages, int stages_per_split, void* __restrict__ y,
                unsigned int* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Layout L(stages, n_tok);
  Barriers& bar = *reinterpret_cast<Barriers*>(base + L.bar_off);
  const uint32_t sbase = smem_addr(base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  static_assert(kDqWarps == 8, "chunk split assumes two warps per TMEM quarter");
  const int64_t n0 = (int64_t)blockIdx.x * BM;
  const int64_t m0 = (int64_t)blockIdx.z * n_tok;
  const int nchunk = (int)(K / kChunkK);
  const int nstage_total = (nchunk + 3) / 4;
  const int st_begin = blockIdx.y * stages_per_split;
  const int st_end = min(st_begin + stages_per_split, nstage_total);
  const int nst = max(0, st_end - st_begin);
  const int64_t ct = K / 64;  // scale column tiles per row tile

  // The producer thread initialises every barrier and starts the first
  // stages' copies right away, while warp 0 allocates TMEM.
  const bool producer = warp == kProducerWarp && lane == 0;
  int issued = 0;
  auto issue_stage = [&](int i) {
    const int s = i % stages;
    const int st = st_begin + i;
    const int chunks = min(4, nchunk - 4 * st);
    mbar_arrive_expect_tx(&bar.full[s], kCodesBytes + chunks * (kScaleTileBytes + L.x_bytes));
    tma_load_2d(base + L.codes(s), &tmap_codes, st * (kStageK / 2), (int)n0, &bar.full[s]);
    bulk_load(base + L.sf(s), smma + ((n0 / 128) * ct + 4 * st) * kScaleTileBytes, chunks * kScaleTileBytes,
              &bar.full[s]);
    for (int q = 0; q < chunks; ++q)
      tma_load_2d(base + L.x(s, q), &tmap_x, st * kStageK + q * kChunkK, (int)m0, &bar.full[s]);
  };
  if (producer) {
    prefetch_tmap(&tmap_codes);
    prefetch_tmap(&tmap_x);
    for (int s = 0; s < stages; ++s) {
      mbar_init(&bar.full[s], 1);
      mbar_init(&bar.empty[s], 2);  // one commit per MMA issuer
    }
    for (int a = 0; a < kASlots; ++a) {
      mbar_init(&bar.a_full[a], 4);  // one arrival per dequant warp of a chunk's warp set
      mbar_init(&bar.a_free[a], 1);
    }
    mbar_init(&bar.acc[0], 1);
    mbar_init(&bar.acc[1], 1);
    fence_mbar_init();
    griddep_wait();  // inputs may be written by the previous kernel in the stream
    for (; issued < min(nst, stages); ++issued) issue_stage(issued);
  }
  if (warp == 0) tmem_alloc(&bar.tmem_base, kTmemCols);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = bar.tmem_base;
  bool failed = false;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      // ---------------- TMA producer: remaining stages ----------------
      for (int i = issued; i < nst; ++i) {
        if (!mbar_wait(&bar.empty[i % stages], (uint32_t)(i / stages - 1) & 1u)) {
          failed = true;
          break;
        }
        issue_stage(i);
      }
      for (int i = max(0, nst - stages); i < nst && !failed; ++i)
        if (!mbar_wait(&bar.full[i % stages], (uint32_t)(i / stages) & 1u)) failed = true;
    }
  } else if (warp >= kMmaWarp) {
    if (lane == 0) {
      // ---------------- MMA issuers (chunks of one parity each) ----------------
      const int par = warp - kMmaWarp;
      const uint32_t idesc = idesc_bf16(n_tok);
      const uint32_t dacc = tmem + kAccCol + 64u * par;
      int c = 0;
      for (int i = 0; i < nst && !failed; ++i) {
        const int s = i % stages;
        if (!mbar_wait(&bar.full[s], (uint32_t)(i / stages) & 1u)) {
          failed = true;
          break;
        }
        const int chunks = min(4, nchunk - 4 * (st_begin + i));
        for (int q = 0; q < chunks && !failed; ++q, ++c) {
          if ((c & 1) != par) continue;
          const int slot = c % kASlots;
          if (!mbar_wait(&bar.a_full[slot], (uint32_t)(c / kASlots) & 1u)) {
            failed = true;
            break;
          }
          fence_after_sync();
          const uint64_t bdesc = smem_desc(sbase + L.x(s, q), 0, 1024, 2);
          const uint32_t a = tmem + kACol + 32u * slot;
          mma_bf16_ts(dacc, a, bdesc, idesc, c >= 2);
          mma_bf16_ts(dacc, a + 8u, bdesc + 2ull, idesc, 1u);
          mma_bf16_ts(dacc, a + 16u, bdesc + 4ull, idesc, 1u);
          mma_bf16_ts(dacc, a + 24u, bdesc + 6ull, idesc, 1u);
          commit(&bar.a_free[slot]);
        }
        commit(&bar.empty[s]);
      }
      // the stage buffers are released when both issuers are done with them:
      // each issuer commits to the stage's empty barrier (count 2)
      if (!failed) commit(&bar.acc[par]);
      griddep_launch_dependents();
    }
  } else {
    // ---------------- dequantisation (warps 0-7, one weight row per thread) ----------------
    const int row = threadIdx.x & 127;  // TMEM lane and tile row
    const int parity = warp >> 2;       // this warp takes the chunks c with c % 2 == parity
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    int c = 0;
    for (int i = 0; i < nst && !failed; ++i) {
      const int s = i % stages;
      if (!mbar_wait(&bar.full[s], (uint32_t)(i / stages) & 1u)) {
        failed = true;
        break;
      }
      const int chunks = min(4, nchunk - 4 * (st_begin + i));
      const uint8_t* crow = base + L.codes(s) + row * 128;
      const uint8_t* srow = base + L.sf(s) + (row & 31) * 16 + (row >> 5) * 4;
      for (int q = 0; q < chunks; ++q, ++c) {
        if ((c & 1) != parity) continue;
        const int slot = c % kASlots;
        if (c >= kASlots && !mbar_wait(&bar.a_free[slot], (uint32_t)(c / kASlots - 1) & 1u)) {
          failed = true;
          break;
        }
        // 32 code bytes of this row: two 16-byte units, 128-byte swizzle
        const uint4 u0 = *reinterpret_cast<const uint4*>(crow + (((2 * q) ^ (row & 7)) << 4));
        const uint4 u1 = *reinterpret_cast<const uint4*>(crow + (((2 * q + 1) ^ (row & 7)) << 4));
        const uint32_t sc = *reinterpret_cast<const uint32_t*>(srow + q * kScaleTileBytes);
        uint32_t w[32];
        const uint32_t cw[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
        for (int b = 0; b < 4; ++b) {  // 16-element block b of the chunk
          const uint32_t s2 = scale_pair((sc >> (8 * b)) & 0xFFu);
          dequant8(cw[2 * b], s2, w + 8 * b);
          dequant8(cw[2 * b + 1], s2, w + 8 * b + 4);
        }
        tmem_st_32x32b_x32(tmem + lane_base + kACol + 32u * slot, w);
        tmem_wait_st();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.a_full[slot]);
      }
    }
  }
  __syncwarp();

  // ---------------- epilogue ----------------
  const bool ks1 = gridDim.y == 1;
  float* red = reinterpret_cast<float*>(base);  // [n_tok][BM] partial tile (split-K)
  bool acc_ok = true;
  if (warp < 4) {
    acc_ok = __all_sync(0xffffffffu, !failed && (nst == 0 || (mbar_wait(&bar.acc[0], 0) && mbar_wait(&bar.acc[1], 0))));
    fence_after_sync();
    const int row = threadIdx.x;
    const int64_t n = n0 + row;
    const float alpha = __fmul_rn(*ts_ptr, 128.0f);
    // chunks this CTA accumulated: the odd accumulator is live from 2 on
    const int nch = nst > 0 ? min(4 * st_end, nchunk) - 4 * st_begin : 0;
    for (int j = 0; j < n_tok; j += 16) {
      uint32_t v[16];
      if (acc_ok && nch > 0) {
        tmem_ld_32x32b_x16(tmem + ((uint32_t)(warp * 32) << 16) + kAccCol + j, v);
        if (nch > 1) {
          uint32_t v1[16];
          tmem_ld_32x32b_x16(tmem + ((uint32_t)(warp * 32) << 16) + kAccCol + 64u + j, v1);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) + __uint_as_float(v1[e]));
        } else {
          tmem_wait_ld();
        }
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = 0u;
      }
      if (ks1) {
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int64_t m = m0 + j + e;
          if (m < M && n < N) store_out<kF32>(y, m * N + n, __uint_as_float(v[e]) * alpha);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) red[(j + e) * BM + row] = __uint_as_float(v[e]);
      }
    }
    if (!acc_ok && lane == 0) atomicOr(status, kStatusTimeout);
  }
  if (!ks1) {
    // cluster-wide reduction: CTA `rank` sums one slice of the tile over all
    // CTAs of the cluster, in rank order, and stores it
    cluster_sync_all();
    const uint32_t ks = gridDim.y, rank = cluster_ctarank();
    const int nvec = n_tok * BM / 4;
    const int lo = (int)((rank * (uint32_t)nvec) / ks), hi = (int)(((rank + 1) * (uint32_t)nvec) / ks);
    const float alpha = __fmul_rn(*ts_ptr, 128.0f);
    for (int i = lo + threadIdx.x; i < hi; i += kThreads) {
      float4 acc = ld_dsmem_f4(sbase + 16u * i, 0);
      for (uint32_t q = 1; q < ks; ++q) {
        const float4 v = ld_dsmem_f4(sbase + 16u * i, q);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      const int tk = (4 * i) / BM, nl = (4 * i) % BM;
      const int64_t m = m0 + tk, n = n0 + nl;
      if (m < M) {
        const float o[4] = {acc.x * alpha, acc.y * alpha, acc.z * alpha, acc.w * alpha};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (n + e < N) store_out<kF32>(y, m * N + n + e, o[e]);
      }
    }
    cluster_sync_all();
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
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

// Row-major 2-D tensor, boxes of [box_rows, 128 bytes], 128-byte swizzle,
// zero fill outside.
bool make_map(CUtensorMap* map, CUtensorMapDataType dt, uint32_t elem_bytes, const void* base, uint64_t rows,
              uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * elem_bytes};
  cuuint32_t box[2] = {128u / elem_bytes, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_gemm_w4a16(const void* x, int64_t M, const uint8_t* codes, const uint8_t* scales_mma,
                              const float* ts, int64_t N, int64_t K, void* y, bool out_f32,
                              unsigned int* status, int num_sms, cudaStream_t stream) {
  if (M <= 0) return cudaSuccess;
  if (K % 64 != 0 || N > INT32_MAX || M > INT32_MAX) return cudaErrorNotSupported;
  const int n_tok = (int)std::min<int64_t>(kMaxTok, (M + 15) / 16 * 16);
  const int64_t groups = (M + n_tok - 1) / n_tok;
  const int64_t tiles = (N + BM - 1) / BM;
  const int nchunk = (int)(K / kChunkK);
  const int nstage_total = (nchunk + 3) / 4;
  int64_t ks = (2 * (int64_t)num_sms + tiles * groups - 1) / (tiles * groups);
  ks = std::max<int64_t>(1, std::min<int64_t>({ks, (int64_t)kMaxCluster, (int64_t)nstage_total}));
  const int sps = (int)((nstage_total + ks - 1) / ks);
  ks = (nstage_total + sps - 1) / sps;
  if (groups > 65535) return cudaErrorNotSupported;
  // as many stages as the split needs (2..4), within the 227 KB of shared memory
  int stages = std::max(2, std::min(4, sps));
  while (stages > 2 && Layout(stages, n_tok).total > 227u * 1024u) --stages;
  const Layout L(stages, n_tok);
  // Each CTA allocates kTmemCols of the SM's 512 TMEM columns, and TMEM is not
  // a resource the block scheduler counts: request enough shared memory that
  // at most 512 / kTmemCols = 2 CTAs are ever resident on one SM, so that
  // tcgen05.alloc never has to wait for another CTA (which, with clusters,
  // could wait in turn on this one).
  static_assert(kTmemCols * 2 <= 512, "TMEM per SM");
  const uint32_t smem = std::max<uint32_t>(L.total, kSmemFor2PerSm);
  CUtensorMap mc, mx;
  if (!make_map(&mc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, codes, (uint64_t)N, (uint64_t)K / 2, BM) ||
      !make_map(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, (uint64_t)M, (uint64_t)K, (uint32_t)n_tok))
    return cudaErrorInvalidValue;
  auto kern = out_f32 ? w4a16_tc_kernel<true> : w4a16_tc_kernel<false>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)tiles, (unsigned)ks, (unsigned)groups);
  cfg.blockDim = dim3(kThreads);
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
  return cudaLaunchKernelEx(&cfg, kern, mc, mx, scales_mma, ts, M, N, K, n_tok, stages, sps, y, status);
}

}  // namespace nvfp4
