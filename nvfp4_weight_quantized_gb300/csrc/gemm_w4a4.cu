// gemm_w4a4.cu -- NVFP4 x NVFP4 GEMM on the 5th-generation tensor cores.
//
// The large-M path of "SOAR 2026 Recap ...", section "1. Quantization and GEMM
// dispatch": activations quantised online to NVFP4, then a GEMM that natively
// issues the block-scaled FP4 MMA.  On sm_103a that instruction is
// tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X: E2M1 operands packed
// two per byte, one UE4M3 scale per 16 elements along K, fp32 accumulation in
// tensor memory (TMEM).
//
// One CTA computes a 128 x 256 output tile (A rows = tokens, B rows = weight
// rows) with 4 warps:
//   warp 0, one lane  -- producer: per 256-wide K stage, TMA loads of the A and
//                        B code tiles (128-byte swizzle) and bulk copies of the
//                        matching scale tiles (already in the MMA tiling);
//   warp 1, one lane  -- MMA issuer: tcgen05.cp of the scales into TMEM, four
//                        K=64 MMAs per stage, tcgen05.commit to free the stage;
//   all 4 warps       -- epilogue: tcgen05.ld of the accumulator, times
//                        ts_a * ts_w, convert, store.
// A 4-stage shared-memory ring keeps TMA, the MMAs and the next loads in
// flight together.  Every mbarrier wait is bounded; a wait that runs out sets
// the library's status word (NVFP4_ERR_TIMEOUT) and the CTA winds down.
#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace nvfp4 {

namespace {

using namespace sm100;

constexpr int BM = 128;             // tokens per tile (MMA M)
constexpr int BN = 256;             // weight rows per tile (MMA N)
constexpr int BK = 256;             // FP4 elements per stage (128 bytes per row)
constexpr int kStages = 4;
constexpr int kThreads = 128;
constexpr int kABytes = BM * BK / 2;                          // 16 KB
constexpr int kBBytes = BN * BK / 2;                          // 32 KB
constexpr int kSfaBytes = (BM / 128) * (BK / 64) * kScaleTileBytes;  // 2 KB
constexpr int kSfbBytes = (BN / 128) * (BK / 64) * kScaleTileBytes;  // 4 KB
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 0;                       // 256 fp32 columns
constexpr uint32_t kSfaCol = 256;                     // 16 columns per stage
constexpr uint32_t kSfbCol = kSfaCol + 16 * kStages;  // 32 columns per stage
static_assert(kSfbCol + 32 * kStages <= kTmemCols, "TMEM budget");

struct __align__(1024) Smem {
  uint8_t a[kStages][kABytes];
  uint8_t b[kStages][kBBytes];
  uint8_t sfa[kStages][kSfaBytes];
  uint8_t sfb[kStages][kSfbBytes];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t acc;
  uint32_t tmem_base;
};

// Instruction descriptor for kind::mxf4nvf4: A and B E2M1 (format code 1 in
// bits 7-9 and 10-12), both K-major, N >> 3 in bits 17-22, scale type UE4M3
// (bit 23 = 0), M >> 7 in bits 27-28, scale-factor ids 0, dense.
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 7) << 27);

template <bool kF32>
__device__ __forceinline__ void store_row32(void* y, int64_t row_off, int64_t n, int64_t N, const uint32_t (&v)[32],
                                            float alpha, bool vec_ok) {
  float f[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]) * alpha;
  if (kF32) {
    float* out = static_cast<float*>(y) + row_off + n;
    if (vec_ok && n + 32 <= N) {
#pragma unroll
      for (int i = 0; i < 32; i += 4) *reinterpret_cast<float4*>(out + i) = make_float4(f[i], f[i + 1], f[i + 2], f[i + 3]);
    } else {
      for (int i = 0; i < 32 && n + i < N; ++i) out[i] = f[i];
    }
  } else {
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(y) + row_off + n;
    if (vec_ok && n + 32 <= N) {
#pragma unroll
      for (int i = 0; i < 32; i += 8) {
        uint4 p;
        __nv_bfloat162 h0 = __floats2bfloat162_rn(f[i], f[i + 1]);
        __nv_bfloat162 h1 = __floats2bfloat162_rn(f[i + 2], f[i + 3]);
        __nv_bfloat162 h2 = __floats2bfloat162_rn(f[i + 4], f[i + 5]);
        __nv_bfloat162 h3 = __floats2bfloat162_rn(f[i + 6], f[i + 7]);
        p.x = *reinterpret_cast<uint32_t*>(&h0);
        p.y = *reinterpret_cast<uint32_t*>(&h1);
        p.z = *reinterpret_cast<uint32_t*>(&h2);
        p.w = *reinterpret_cast<uint32_t*>(&h3);
        *reinterpret_cast<uint4*>(out + i) = p;
      }
    } else {
      for (int i = 0; i < 32 && n + i < N; ++i) out[i] = __float2bfloat16_rn(f[i]);
    }
  }
}

template <bool kF32>
__global__ void __launch_bounds__(kThreads, 1)
w4a4_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
            const uint8_t* __restrict__ a_smma, const uint8_t* __restrict__ b_smma,
            const float* __restrict__ a_ts, const float* __restrict__ b_ts, int64_t M, int64_t N, int64_t K,
            void* __restrict__ y, unsigned int* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t m_tile = blockIdx.y, n_tile = blockIdx.x;
  const int64_t m0 = m_tile * BM, n0 = n_tile * BN;
  const int kb64 = (int)(K / 64);                 // 64-wide K blocks = scale column tiles per row tile
  const int kt = (kb64 + 3) / 4;                  // K stages
  const int64_t b_row_tiles = (N + 127) / 128;    // row tiles present in the weight scale tiling
  const int64_t sfb_left = b_row_tiles - n0 / 128;
  const int nsfb = sfb_left < 2 ? (int)sfb_left : 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    mbar_init(&sm.acc, 1);
    fence_mbar_init();
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
  }
  if (warp == 1) tmem_alloc(&sm.tmem_base, kTmemCols);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = sm.tmem_base;
  bool failed = false;

  if (warp == 0 && lane == 0) {
    // ---------------- producer ----------------
    griddep_wait();  // inputs may be written by the previous kernel in the stream
    for (int ks = 0; ks < kt; ++ks) {
      const int s = ks % kStages;
      const uint32_t round = (uint32_t)(ks / kStages);
      if (ks >= kStages && !mbar_wait(&sm.empty[s], (round - 1) & 1u)) {
        failed = true;
        break;
      }
      const int kk_n = min(4, kb64 - 4 * ks);
      const uint32_t sf_bytes = (uint32_t)kk_n * kScaleTileBytes;
      mbar_arrive_expect_tx(&sm.full[s], kABytes + kBBytes + sf_bytes * (1 + nsfb));
      tma_load_2d(sm.a[s], &tmap_a, ks * (BK / 2), (int)m0, &sm.full[s]);
      tma_load_2d(sm.b[s], &tmap_b, ks * (BK / 2), (int)n0, &sm.full[s]);
      bulk_load(sm.sfa[s], a_smma + (m_tile * kb64 + 4 * ks) * kScaleTileBytes, sf_bytes, &sm.full[s]);
      for (int rt = 0; rt < nsfb; ++rt)
        bulk_load(sm.sfb[s] + rt * (kSfbBytes / 2), b_smma + ((n0 / 128 + rt) * kb64 + 4 * ks) * kScaleTileBytes,
                  sf_bytes, &sm.full[s]);
    }
    // let every load this thread issued land before the CTA can exit
    for (int ks = max(0, kt - kStages); ks < kt && !failed; ++ks)
      if (!mbar_wait(&sm.full[ks % kStages], (uint32_t)(ks / kStages) & 1u)) failed = true;
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    for (int ks = 0; ks < kt; ++ks) {
      const int s = ks % kStages;
      if (!mbar_wait(&sm.full[s], (uint32_t)(ks / kStages) & 1u)) {
        failed = true;
        break;
      }
      fence_after_sync();
      const int kk_n = min(4, kb64 - 4 * ks);
      const uint32_t sfa_t = tmem + kSfaCol + 16u * s, sfb_t = tmem + kSfbCol + 32u * s;
      const uint32_t sfa_s = smem_addr(sm.sfa[s]), sfb_s = smem_addr(sm.sfb[s]);
      for (int kk = 0; kk < kk_n; ++kk) {
        cp_32x128b_warpx4(sfa_t + 4 * kk, smem_desc(sfa_s + kk * kScaleTileBytes, 0, 128, 0));
        for (int rt = 0; rt < nsfb; ++rt)
          cp_32x128b_warpx4(sfb_t + 8 * kk + 4 * rt,
                            smem_desc(sfb_s + rt * (kSfbBytes / 2) + kk * kScaleTileBytes, 0, 128, 0));
      }
      const uint64_t adesc = smem_desc(smem_addr(sm.a[s]), 0, 1024, 2);
      const uint64_t bdesc = smem_desc(smem_addr(sm.b[s]), 0, 1024, 2);
      for (int kk = 0; kk < kk_n; ++kk) {
        // advancing the start address by 32 bytes selects the next 64 FP4
        // elements inside the 128-byte swizzle atom
        mma_mxf4nvf4(tmem + kAccCol, adesc + 2ull * kk, bdesc + 2ull * kk, kIdesc, sfa_t + 4 * kk, sfb_t + 8 * kk,
                     (ks | kk) != 0);
      }
      commit(&sm.empty[s]);
    }
    if (!failed) commit(&sm.acc);
    griddep_launch_dependents();
  }
  __syncwarp();

  // ---------------- epilogue ----------------
  // warp-uniform, since tcgen05.ld is a warp-collective instruction
  const bool acc_ok = __all_sync(0xffffffffu, !failed && mbar_wait(&sm.acc, 0));
  fence_after_sync();
  if (acc_ok) {
    const float alpha = __fmul_rn(*a_ts, *b_ts);
    const int64_t row = m0 + warp * 32 + lane;
    const bool vec_ok = kF32 ? (N % 4 == 0) : (N % 8 == 0);
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      uint32_t v[32];
      tmem_ld_32x32b_x32(tmem + ((uint32_t)(warp * 32) << 16) + kAccCol + c, v);
      tmem_wait_ld();
      if (row < M && n0 + c < N) store_row32<kF32>(y, row * N, n0 + c, N, v, alpha, vec_ok);
    }
  } else if (lane == 0) {
    atomicOr(status, kStatusTimeout);
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 1) {
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

}  // namespace

cudaError_t launch_gemm_w4a4(const uint8_t* a_codes, const uint8_t* a_scales_mma, const float* a_ts, int64_t M,
                             const uint8_t* w_codes, const uint8_t* w_scales_mma, const float* w_ts, int64_t N,
                             int64_t K, void* y, bool out_f32, unsigned int* status, int num_sms,
                             cudaStream_t stream) {
  (void)num_sms;
  if (M <= 0) return cudaSuccess;
  if (K < BK || K % 64 != 0 || (M + BM - 1) / BM > 65535 || M > INT32_MAX || N > INT32_MAX)
    return cudaErrorNotSupported;
  CUtensorMap ma, mb;
  if (!make_map(&ma, a_codes, (uint64_t)M, (uint64_t)K / 2, BM) ||
      !make_map(&mb, w_codes, (uint64_t)N, (uint64_t)K / 2, BN))
    return cudaErrorInvalidValue;
  const size_t smem = sizeof(Smem) + 1024;
  auto kern = out_f32 ? w4a4_kernel<true> : w4a4_kernel<false>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((N + BN - 1) / BN), (unsigned)((M + BM - 1) / BM));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, ma, mb, a_scales_mma, w_scales_mma, a_ts, w_ts, M, N, K, y, status);
}

}  // namespace nvfp4
