// fp4_rate.cu -- the dense block-scaled FP4 tensor-core rate of this GPU,
// measured with the same instruction stream as the W4A4 CTA-pair kernel but
// no memory traffic: the denominator of the W4A4 roofline fraction.
//
// "SOAR 2026 Recap ...", section "1. Quantization and GEMM dispatch", names
// the NVFP4 MMA as the W4A4 path's engine; the pages give no rate for it, and
// the datasheet figure is not a measurement.  Each CTA pair (one CTA per SM)
// issues `iters` x 4 MMAs of 256 x 256 x 64 (tcgen05.mma.cta_group::2
// .kind::mxf4nvf4.block_scale.scale_vec::4X, zero operands in shared memory,
// zero UE4M3 scales in tensor memory, the pair kernel's descriptors) back to
// back from one thread, then one commit; the caller times the launch.  Every
// wait is bounded.
#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace nvfp4 {

namespace {

using namespace sm100;

constexpr int kRateThreads = 128;       // four warps: one per 32-lane TMEM sub-partition
constexpr uint32_t kRateTmemCols = 512;
constexpr uint32_t kRateSfCol = 256;    // scale columns after the 256 accumulator columns
// kind::mxf4nvf4, E2M1 x E2M1, K-major, N = 256 (bits 17-22), UE4M3 scales,
// M = 256 across the pair (M >> 7 in bits 27-28)
constexpr uint32_t kRateIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(256 >> 3) << 17) | (2u << 27);
constexpr size_t kRateSmem = 120u * 1024u;  // more than half an SM: one CTA (and its 512 TMEM columns) per SM

struct __align__(1024) RateSmem {
  uint8_t a[128 * 128];  // this CTA's 128 A rows of one 256-wide K stage (128-byte swizzle)
  uint8_t b[128 * 128];  // and its 128 B rows
  uint64_t done;
  uint32_t tmem_base;
};

__global__ void __launch_bounds__(kRateThreads, 1)
fp4_mma_rate_kernel(int iters, unsigned long long* __restrict__ cycles, unsigned int* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  RateSmem& sm = *reinterpret_cast<RateSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t rank = cluster_rank();
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < (int)(sizeof(sm.a) + sizeof(sm.b)) / 16; i += kRateThreads)
    reinterpret_cast<uint4*>(sm.a)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    mbar_init(&sm.done, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc_pair(&sm.tmem_base, kRateTmemCols);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // zeros visible to the MMA's reads
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = sm.tmem_base;
  {  // zero scale factors in the 64 scale columns of every lane
    uint32_t z[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) z[i] = 0u;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_st_x16(tmem + lane_base + kRateSfCol + 16 * c, z);
    tmem_wait_st();
  }
  fence_before_sync();
  __syncthreads();
  cluster_sync();  // both CTAs' operands, scales and barrier are in place
  fence_after_sync();
  bool failed = false;
  if (threadIdx.x == 0) {
    long long t0 = clock64();
    if (rank == 0) {
      const uint64_t adesc = smem_desc(smem_addr(sm.a), 0, 1024, 2), bdesc = smem_desc(smem_addr(sm.b), 0, 1024, 2);
      for (int it = 0; it < iters; ++it)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_mxf4nvf4_pair(tmem, adesc + 2ull * kk, bdesc + 2ull * kk, kRateIdesc, tmem + kRateSfCol + 4 * kk,
                            tmem + kRateSfCol + 16 + 8 * kk, 1u);
      commit_pair(&sm.done, (uint16_t)3u);
    }
    // both CTAs: the pair's MMAs have completed
    if (!mbar_wait(&sm.done, 0u)) failed = true;
    if (rank == 0) cycles[blockIdx.x / 2] = (unsigned long long)(clock64() - t0);
    if (failed) atomicOr(status, kStatusTimeout);
  }
  fence_before_sync();
  __syncthreads();
  cluster_sync();
  if (warp == 0) {
    fence_after_sync();
    tmem_dealloc_pair(tmem, kRateTmemCols);
  }
}

}  // namespace

cudaError_t launch_fp4_mma_rate(int iters, unsigned long long* cycles, int max_pairs, int* pairs,
                                unsigned int* status, cudaStream_t stream) {
  *pairs = 0;
  if (iters <= 0 || max_pairs <= 0) return cudaErrorInvalidValue;
  cudaError_t err = cudaFuncSetAttribute(fp4_mma_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kRateSmem);
  if (err != cudaSuccess) return err;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kRateThreads);
  cfg.dynamicSmemBytes = kRateSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(2);
  int n = 0;
  if ((err = cudaOccupancyMaxActiveClusters(&n, fp4_mma_rate_kernel, &cfg)) != cudaSuccess) return err;
  if (n < 1) return cudaErrorNotSupported;
  n = std::min(n, max_pairs);
  cfg.gridDim = dim3((unsigned)(2 * n));
  err = cudaLaunchKernelEx(&cfg, fp4_mma_rate_kernel, iters, cycles, status);
  if (err == cudaSuccess) *pairs = n;
  return err;
}

}  // namespace nvfp4
