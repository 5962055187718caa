// gptq.cu -- GPTQ inside FourOverSix block scales.
//
// "SOAR Weekly Champion Notes 07 ... NVFP4 Quantization Improvements",
// section "03 How we integrated it": each 16-element block's scale is chosen
// first (M=4 or M=6, as nvfp4_quantize_fos does on the original weights) and
// GPTQ's error-compensating quantisation then runs inside that choice.  GPTQ
// quantises the columns of W in order; each column's error, divided by the
// diagonal of U (the upper Cholesky factor of the inverse of the damped
// Hessian H + d I), is spread over the columns not yet quantised along the
// rows of U, at once inside a block of 128 columns and once per block beyond.
//
// The steps are plain kernels in binary32 with one rounding per operation and
// a fixed order (the order is part of the contract: the codes are decided in
// binary32, and an independent implementation taking the same steps must get
// the same bits):
//   gptq_damp_kernel      d = damp * ((sum_k H[k][k], k ascending) / K)
//   gptq_reverse_kernel   A = J (H + d I) J  (J reverses indices)
//   chol_panel_kernel / chol_trail_kernel, right-looking, column j in order:
//                         L[j][j] = sqrt(A[j][j]); L[i][j] = A[i][j] / L[j][j];
//                         A[i][c] = fma(-L[i][j], L[c][j], A[i][c]), j < c <= i
//                         (in 32-column panels: the same operations on every
//                         element in the same order, 2K / 32 launches)
//   trinv_kernel          Linv = L^-1 by columns: x[j] = 1 / L[j][j],
//                         x[i] = -(sum_{k=j}^{i-1} fma(L[i][k], x[k], .)) / L[i][i]
//                         (U = J Linv J, read through reversed indices)
//   gptq_block_kernel     one thread per row: for each column j of the block,
//                         q = e2m1(RN(w / eff)), e = fma(-value(q), eff, w) / U[j][j],
//                         then w[c] = fma(-e, U[j][c], w[c]) for the block's later columns
//   gptq_trail_kernel     w[n][c] -= sum_{j in block} fma(E[n][j], U[j][c], .) (j ascending)
#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

namespace {

constexpr int kBlock = 128;  // GPTQ columns per block
constexpr int kPitch = kBlock + 1;  // shared-memory row pitch (no bank conflicts down a column)

__device__ __forceinline__ float u_at(const float* __restrict__ li, int64_t K, int64_t i, int64_t j) {
  return li[(K - 1 - i) * K + (K - 1 - j)];
}

__global__ void gptq_damp_kernel(const float* __restrict__ H, int64_t K, float damp, float* __restrict__ d_out) {
  if (blockIdx.x != 0 || threadIdx.x != 0) return;
  float s = 0.0f;
  for (int64_t k = 0; k < K; ++k) s = __fadd_rn(s, H[k * K + k]);
  *d_out = __fmul_rn(damp, __fdiv_rn(s, (float)K));
}

__global__ void gptq_reverse_kernel(const float* __restrict__ H, int64_t K, const float* __restrict__ d,
                                    float* __restrict__ A) {
  const float dv = *d;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < K * K; e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = e / K, j = e - i * K;
    const float h = H[(K - 1 - i) * K + (K - 1 - j)];
    A[e] = i == j ? __fadd_rn(h, dv) : h;
  }
}

// Panelled form of the column loop: 32 columns at a time in two launches,
// each element receiving the same fused multiply-adds in the same order.
// chol_panel_kernel: every CTA redundantly factors the panel's top 32 x 32
// block in shared memory (identical arithmetic in every CTA), CTA 0 writes
// it back, and each CTA then finishes its own rows below the panel top:
// for j in the panel, L[i][j] = A[i][j] / p_j, then the panel's later
// columns of the row get fma(-L[i][j], L[c][j], .).
constexpr int kPanel = 32;
constexpr int kPanelRows = 256;  // rows below the top block per CTA (one per thread)

__global__ void __launch_bounds__(kPanelRows)
chol_panel_kernel(float* __restrict__ A, int64_t K, int64_t p0, float* __restrict__ piv,
                  unsigned int* __restrict__ status) {
  __shared__ float top[kPanel][kPanel + 1];
  __shared__ float pv[kPanel];
  const int pw = (int)(K - p0 < kPanel ? K - p0 : kPanel);
  const int t = threadIdx.x;
  for (int e = t; e < pw * pw; e += blockDim.x) {
    const int r = e / pw, c = e - r * pw;
    top[r][c] = A[(p0 + r) * K + p0 + c];
  }
  __syncthreads();
  // the top block, column by column (lower triangle, c <= r)
  for (int j = 0; j < pw; ++j) {
    if (t == 0) {
      const float a = top[j][j];
      if (!(a > 0.0f)) atomicOr(status, kStatusNonfinite);
      pv[j] = __fsqrt_rn(a);
    }
    __syncthreads();
    const float p = pv[j];
    for (int r = j + 1 + t; r < pw; r += blockDim.x) top[r][j] = __fdiv_rn(top[r][j], p);
    __syncthreads();
    for (int e = t; e < pw * pw; e += blockDim.x) {
      const int r = e / pw, c = e - r * pw;
      if (r > j && c > j && c <= r) top[r][c] = __fmaf_rn(-top[r][j], top[c][j], top[r][c]);
    }
    __syncthreads();
  }
  if (blockIdx.x == 0) {
    for (int e = t; e < pw * pw; e += blockDim.x) {
      const int r = e / pw, c = e - r * pw;
      if (c < r) A[(p0 + r) * K + p0 + c] = top[r][c];
      else if (c == r) piv[p0 + r] = pv[r];
    }
  }
  // rows below the top block
  const int64_t i = p0 + pw + (int64_t)blockIdx.x * kPanelRows + t;
  if (i >= K) return;
  float w[kPanel];
#pragma unroll
  for (int c = 0; c < kPanel; ++c) w[c] = c < pw ? A[i * K + p0 + c] : 0.0f;
#pragma unroll
  for (int j = 0; j < kPanel; ++j) {
    if (j < pw) {
      w[j] = __fdiv_rn(w[j], pv[j]);
#pragma unroll
      for (int c = j + 1; c < kPanel; ++c)
        if (c < pw) w[c] = __fmaf_rn(-w[j], top[c][j], w[c]);
    }
  }
#pragma unroll
  for (int c = 0; c < kPanel; ++c)
    if (c < pw) A[i * K + p0 + c] = w[c];
}

// Elements (i, c), pend <= c <= i < K: the panel's updates in column order,
// 32 columns x 8 rows per CTA with the panel rows of those columns and rows
// in shared memory.
__global__ void __launch_bounds__(256)
chol_trail_kernel(float* __restrict__ A, int64_t K, int64_t p0, int pw) {
  __shared__ float lc[32][kPanel + 1], lr[8][kPanel + 1];
  const int64_t pend = p0 + pw;
  const int64_t c0 = pend + (int64_t)blockIdx.x * 32, i0 = pend + (int64_t)blockIdx.y * 8;
  if (i0 + 7 < c0) return;  // wholly above the diagonal
  const int tx = threadIdx.x, ty = threadIdx.y, t = ty * 32 + tx;
  for (int e = t; e < 32 * pw; e += 256) {
    const int r = e / pw, q = e - r * pw;
    lc[r][q] = c0 + r < K ? A[(c0 + r) * K + p0 + q] : 0.0f;
  }
  for (int e = t; e < 8 * pw; e += 256) {
    const int r = e / pw, q = e - r * pw;
    lr[r][q] = i0 + r < K ? A[(i0 + r) * K + p0 + q] : 0.0f;
  }
  __syncthreads();
  const int64_t c = c0 + tx, i = i0 + ty;
  if (i >= K || c > i) return;
  float v = A[i * K + c];
  for (int q = 0; q < pw; ++q) v = __fmaf_rn(-lr[ty][q], lc[tx][q], v);
  A[i * K + c] = v;
}

__global__ void chol_diag_kernel(float* __restrict__ A, int64_t K, const float* __restrict__ piv) {
  for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < K; j += (int64_t)gridDim.x * blockDim.x)
    A[j * K + j] = piv[j];
}

// Inverse of the lower factor: a CTA (one warp) owns kInvCols consecutive
// columns j0 .. and keeps their entries x[k], k >= j0, in shared memory
// ([k][lane], conflict-free).  For each row i all 32 lanes first copy
// L[i][j0 .. i] into shared memory (coalesced), then the kInvCols lanes take
// their dot products from there.  A lane starts its sum at k = j0 instead of
// its own j: the extra terms are fma(L[i][k], 0, s) = s exactly (x[k] = 0 for
// k < j; s starts at +0), so every column gets the bits of the sum taken from
// k = j.
constexpr int kInvCols = 4;

__global__ void __launch_bounds__(32) trinv_kernel(const float* __restrict__ L, int64_t K, float* __restrict__ li) {
  extern __shared__ float xs[];  // [(K - j0)][kInvCols], then row [K - j0]
  const int lane = threadIdx.x;
  const int64_t j0 = (int64_t)blockIdx.x * kInvCols, j = j0 + lane;
  float* row = xs + (K - j0) * kInvCols;
  for (int64_t e = lane; e < (K - j0) * kInvCols; e += 32) xs[e] = 0.0f;
  const bool mine = lane < kInvCols && j < K;
  for (int64_t i = j0; i < K; ++i) {
    {  // four loads in flight per lane
      const float* src = L + i * K;
      int64_t k = j0 + lane;
      for (; k + 96 <= i; k += 128) {
        const float v0 = src[k], v1 = src[k + 32], v2 = src[k + 64], v3 = src[k + 96];
        row[k - j0] = v0;
        row[k + 32 - j0] = v1;
        row[k + 64 - j0] = v2;
        row[k + 96 - j0] = v3;
      }
      for (; k <= i; k += 32) row[k - j0] = src[k];
    }
    __syncwarp();
    if (mine && i >= j) {
      float x;
      if (i == j) {
        x = __fdiv_rn(1.0f, row[i - j0]);
      } else {
        float s = 0.0f;
#pragma unroll 8
        for (int64_t k = j0; k < i; ++k) s = __fmaf_rn(row[k - j0], xs[(k - j0) * kInvCols + lane], s);
        x = __fdiv_rn(-s, row[i - j0]);
      }
      xs[(i - j0) * kInvCols + lane] = x;
      li[i * K + j] = x;
    }
    __syncwarp();  // the row buffer is rewritten next
  }
}

__global__ void bf16_to_f32_kernel(const __nv_bfloat16* __restrict__ x, int64_t n, float* __restrict__ y) {
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x)
    y[e] = __bfloat162float(x[e]);
}

// One block of columns [b0, b0 + bw) for 128 rows per CTA (one per thread),
// the block's U in shared memory.
__global__ void __launch_bounds__(kBlock)
gptq_block_kernel(float* __restrict__ wc, int64_t N, int64_t K, int64_t b0, int bw, const float* __restrict__ li,
                  const uint8_t* __restrict__ scales, const float* __restrict__ ts_ptr, uint8_t* __restrict__ codes,
                  float* __restrict__ E) {
  extern __shared__ float sm[];
  float* ub = sm;                    // [bw][kPitch]
  float* wt = sm + kBlock * kPitch;  // [128 rows][kPitch]
  const int t = threadIdx.x;
  for (int e = t; e < bw * bw; e += kBlock) {
    const int a = e / bw, b = e - a * bw;
    ub[a * kPitch + b] = u_at(li, K, b0 + a, b0 + b);
  }
  const int64_t n0 = (int64_t)blockIdx.x * kBlock;
  for (int e = t; e < kBlock * bw; e += kBlock) {  // coalesced along the columns
    const int r = e / bw, c = e - r * bw;
    wt[r * kPitch + c] = n0 + r < N ? wc[(n0 + r) * K + b0 + c] : 0.0f;
  }
  __syncthreads();
  const int64_t n = n0 + t;
  if (n < N) {
    const float ts = *ts_ptr;
    float* w = wt + t * kPitch;
    uint32_t lo = 0;
    for (int jj = 0; jj < bw; ++jj) {
      const int64_t j = b0 + jj;
      const float eff = __fmul_rn(e4m3_to_f32(scales[n * (K / 16) + j / 16]), ts);
      const float x = w[jj];
      uint32_t q;
      float d;
      if (eff == 0.0f) {
        q = signbit(x) ? 8u : 0u;
        d = x;
      } else {
        q = cvt_e2m1x2(0.0f, __fdiv_rn(x, eff)) & 15u;
        const float mag = e2m1_mag_to_f32(q & 7u);
        d = __fmaf_rn(-(q & 8u ? -mag : mag), eff, x);
      }
      const float err = __fdiv_rn(d, ub[jj * kPitch + jj]);
      E[n * kBlock + jj] = err;
      for (int c = jj + 1; c < bw; ++c) w[c] = __fmaf_rn(-err, ub[jj * kPitch + c], w[c]);
      if (jj & 1) codes[n * (K / 2) + j / 2] = (uint8_t)(lo | (q << 4));
      else lo = q;
    }
  }
}

// Columns after the block: 16 x 16 (row, column) tiles, the block's errors
// and U rows read through L1.
__global__ void gptq_trail_kernel(float* __restrict__ wc, int64_t N, int64_t K, int64_t b0, int bw,
                                  const float* __restrict__ E, const float* __restrict__ li) {
  const int64_t c = b0 + bw + (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t n = (int64_t)blockIdx.y * blockDim.y + threadIdx.y;
  if (c >= K || n >= N) return;
  float s = 0.0f;
  for (int jj = 0; jj < bw; ++jj) s = __fmaf_rn(E[n * kBlock + jj], u_at(li, K, b0 + jj, c), s);
  wc[n * K + c] = __fsub_rn(wc[n * K + c], s);
}

}  // namespace

int64_t gptq_max_k() { return (int64_t)(227 * 1024) / ((kInvCols + 1) * (int64_t)sizeof(float)) / 16 * 16; }

size_t gptq_workspace_bytes(int64_t N, int64_t K) {
  auto a256 = [](size_t b) { return (b + 255) & ~(size_t)255; };
  return 2 * a256((size_t)K * K * 4) + a256((size_t)N * K * 4) + a256((size_t)N * kBlock * 4) + a256((size_t)K * 4) +
         256;
}

// W bf16 [N, K]; H fp32 [K, K]; scales logical [N, K/16] and ts from
// nvfp4_quantize_fos on the same W; codes [N, K/2] overwritten.
cudaError_t launch_gptq(const void* W, int64_t N, int64_t K, const float* H, float damp, const uint8_t* scales,
                        const float* ts, uint8_t* codes, void* workspace, unsigned int* status,
                        cudaStream_t stream) {
  auto a256 = [](size_t b) { return (b + 255) & ~(size_t)255; };
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* A = reinterpret_cast<float*>(ws);
  float* li = reinterpret_cast<float*>(ws + a256((size_t)K * K * 4));
  float* wc = reinterpret_cast<float*>(ws + 2 * a256((size_t)K * K * 4));
  float* E = reinterpret_cast<float*>(ws + 2 * a256((size_t)K * K * 4) + a256((size_t)N * K * 4));
  float* piv = reinterpret_cast<float*>(ws + 2 * a256((size_t)K * K * 4) + a256((size_t)N * K * 4) +
                                        a256((size_t)N * kBlock * 4));
  float* d = piv + a256((size_t)K * 4) / 4;
  cudaError_t err;
  gptq_damp_kernel<<<1, 32, 0, stream>>>(H, K, damp, d);
  gptq_reverse_kernel<<<1024, 256, 0, stream>>>(H, K, d, A);
  for (int64_t p0 = 0; p0 < K; p0 += kPanel) {
    const int pw = (int)std::min<int64_t>(kPanel, K - p0);
    const int64_t below = K - p0 - pw;
    chol_panel_kernel<<<(unsigned)std::max<int64_t>(1, (below + kPanelRows - 1) / kPanelRows), kPanelRows, 0,
                        stream>>>(A, K, p0, piv, status);
    if (below > 0) {
      dim3 blk(32, 8), grid((unsigned)((below + 31) / 32), (unsigned)((below + 7) / 8));
      chol_trail_kernel<<<grid, blk, 0, stream>>>(A, K, p0, pw);
    }
  }
  chol_diag_kernel<<<(unsigned)((K + 255) / 256), 256, 0, stream>>>(A, K, piv);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  if ((err = cudaMemsetAsync(li, 0, (size_t)K * K * 4, stream)) != cudaSuccess) return err;
  const size_t inv_smem = (size_t)K * (kInvCols + 1) * sizeof(float);
  if ((err = cudaFuncSetAttribute(trinv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)inv_smem)) !=
      cudaSuccess)
    return err;
  trinv_kernel<<<(unsigned)((K + kInvCols - 1) / kInvCols), 32, inv_smem, stream>>>(A, K, li);
  bf16_to_f32_kernel<<<1024, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(W), N * K, wc);
  const size_t smem = (size_t)2 * kBlock * kPitch * sizeof(float);
  if ((err = cudaFuncSetAttribute(gptq_block_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
      cudaSuccess)
    return err;
  for (int64_t b0 = 0; b0 < K; b0 += kBlock) {
    const int bw = (int)std::min<int64_t>(kBlock, K - b0);
    gptq_block_kernel<<<(unsigned)((N + kBlock - 1) / kBlock), kBlock, smem, stream>>>(wc, N, K, b0, bw, li,
                                                                                      scales, ts, codes, E);
    const int64_t rest = K - b0 - bw;
    if (rest > 0) {
      dim3 blk(32, 8), grid((unsigned)((rest + 31) / 32), (unsigned)((N + 7) / 8));
      gptq_trail_kernel<<<grid, blk, 0, stream>>>(wc, N, K, b0, bw, E, li);
    }
  }
  return cudaGetLastError();
}

}  // namespace nvfp4
