// kernels.h -- host-side launchers of the NVFP4 kernels (internal to the library).
#pragma once

#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "nvfp4.h"

namespace nvfp4 {

// Maximum number of per-CTA amax partials (sizes the quantiser workspace).
constexpr int kMaxAmaxPartials = 1024;

size_t quant_workspace_bytes();
// Whether launch_quantize uses the single-launch (cooperative) quantiser.
void quantize_set_single_launch(bool on);
bool quantize_get_single_launch();

// Records the text nvfp4_last_error() returns on this thread.
void set_last_error(const char* what);

// Unique id of the CUDA context current on this thread (the runtime's primary
// context of the current device, made current if needed); false on failure.
// Host-side caches of device addresses are keyed by it.
bool current_context_id(unsigned long long* id);

// nvfp4_linear's branch choice for an M-token call on an [N, K] weight.
bool linear_takes_w4a4(int64_t M, int64_t N, int64_t K);
// nvfp4_linear with the branch already chosen (w4a4 false: W4A16), so a
// caller that sized its scratch for one branch runs exactly that branch.
nvfp4_status linear_branch(const void* X, int64_t M, const nvfp4_weight* W, void* Y, int out_dtype,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream, bool w4a4);

// Tensor amax + quantisation (FourOverSix when `fos`, else M=6 only).
cudaError_t launch_quantize(const void* x, int64_t rows, int64_t K, float divisor, bool fos,
                            uint8_t* codes, uint8_t* scales, uint8_t* scales_mma, float* ts,
                            uint8_t* choice, unsigned long long* m4_count, void* workspace,
                            unsigned int* status, int num_sms, cudaStream_t stream);

// W4A16: Y[M, N] = X[M, K] * dequant(W)^T.
cudaError_t launch_gemm_w4a16(const void* x, int64_t M, const uint8_t* codes,
                              const uint8_t* scales_mma, const float* ts, int64_t N, int64_t K,
                              void* y, bool out_f32, unsigned int* status, int num_sms,
                              cudaStream_t stream);

// W4A16 for M <= w4a16_rf_max_tokens(): dequantisation in registers,
// warp-level MMAs.
int w4a16_rf_max_tokens();
cudaError_t launch_gemm_w4a16_rf(const void* x, int64_t M, const uint8_t* codes,
                                 const uint8_t* scales_mma, const float* ts, int64_t N, int64_t K,
                                 void* y, bool out_f32, bool prefetch_w, unsigned int* status,
                                 int num_sms, cudaStream_t stream);

// The same for M <= w4a16_sk_max_tokens() as a persistent split-K kernel
// with the activations resident in shared memory (f16 MMAs).
int w4a16_sk_max_tokens();
cudaError_t launch_gemm_w4a16_sk(const void* x, int64_t M, const uint8_t* codes,
                                 const uint8_t* scales_mma, const float* ts, int64_t N, int64_t K,
                                 void* y, bool out_f32, bool prefetch_w, unsigned int* status,
                                 int num_sms, cudaStream_t stream);

// W4A16 for K % 16 == 0 with K % 64 != 0 (plain loads, CUDA-core fp32
// accumulation; the tensor-core kernels need 64-wide chunks).
cudaError_t launch_gemm_w4a16_any(const void* x, int64_t M, const uint8_t* codes, const uint8_t* scales_mma,
                                  const float* ts, int64_t N, int64_t K, void* y, bool out_f32, int num_sms,
                                  cudaStream_t stream);

// W4A4: block-scaled FP4 tensor-core GEMM.
cudaError_t launch_gemm_w4a4(const uint8_t* a_codes, const uint8_t* a_scales_mma, const float* a_ts,
                             int64_t M, const uint8_t* w_codes, const uint8_t* w_scales_mma,
                             const float* w_ts, int64_t N, int64_t K, void* y, bool out_f32,
                             unsigned int* status, int num_sms, cudaStream_t stream);
// W4A4 on a gate/up weight [2F, K] with silu(G) * U applied in the GEMM's
// epilogue: Y bf16 [M, F].  CTA pairs above 128 tokens (when pairs are
// enabled), single CTAs otherwise.  cudaErrorNotSupported unless
// F % 128 == 0 and the kernel can be resident.
cudaError_t launch_gemm_w4a4_gate_up(const uint8_t* a_codes, const uint8_t* a_scales_mma, const float* a_ts,
                                     int64_t M, const uint8_t* w_codes, const uint8_t* w_scales_mma,
                                     const float* w_ts, int64_t N, int64_t K, void* y, unsigned int* status,
                                     int num_sms, cudaStream_t stream);
// Y [rows_a, rows_b] (bf16, or fp32 when out_f32) = A B^T for bf16 A
// [rows_a, red] and B [rows_b, red] whose rows are pitch_a / pitch_b elements
// apart (multiples of 8), on the CTA-pair tensor-core kernel (tcgen05
// kind::f16, fp32 accumulation).  cudaErrorNotSupported for a bad pitch or
// when no pair can be resident.
cudaError_t launch_gemm_bf16_tn(const void* a, int64_t pitch_a, const void* b, int64_t pitch_b, int64_t rows_a,
                                int64_t rows_b, int64_t red, void* y, bool out_f32, unsigned int* status,
                                cudaStream_t stream);
// Y[m, f] = silu(y2[m, f]) * y2[m, F + f] for y2 fp32 [M, 2F]; Y [M, F].
cudaError_t launch_silu_mul(const float* y2, int64_t M, int64_t F, void* y, bool out_f32, cudaStream_t stream);

// NVFP4 [R, K] (codes, MMA-tiled scales, device tensor scale) -> bf16 [R, K].
cudaError_t launch_dequant_bf16(const uint8_t* codes, const uint8_t* scales_mma, const float* ts, int64_t R,
                                int64_t K, void* out, int num_sms, cudaStream_t stream);
// The straight-through backward of Y = X_hat W_hat^T (qat.cu): dX = dY W_hat
// (bf16 [M, K], skipped if null) and dW = dY^T X_hat (fp32 [N, K], skipped if
// null) for dY bf16 [M, N], W NVFP4 [N, K] and the quantised activations
// [M, K]; workspace of qat_workspace_bytes(M, N, K) (transposed bf16
// operands).
size_t qat_workspace_bytes(int64_t M, int64_t N, int64_t K);
cudaError_t qat_backward(const void* dy, int64_t M, const uint8_t* w_codes, const uint8_t* w_smma, const float* w_ts,
                         int64_t N, int64_t K, const uint8_t* a_codes, const uint8_t* a_smma, const float* a_ts,
                         void* dx, void* dw, void* workspace, unsigned int* status, cudaStream_t stream);

// GPTQ inside FourOverSix scales (see gptq.cu): W bf16 [N, K], H fp32 [K, K],
// scales logical [N, K/16] and ts from the FourOverSix quantiser on W; codes
// [N, K/2] are overwritten.  workspace of gptq_workspace_bytes(N, K).
size_t gptq_workspace_bytes(int64_t N, int64_t K);
int64_t gptq_max_k();  // largest K the triangular inverse's shared memory holds
cudaError_t launch_gptq(const void* W, int64_t N, int64_t K, const float* H, float damp, const uint8_t* scales,
                        const float* ts, uint8_t* codes, void* workspace, unsigned int* status,
                        cudaStream_t stream);

// CTAs per cluster for M > 128: 2 (one pair, cta_group::2 MMAs on 256 x 256
// tiles) or 1 (single CTAs on 128 x 256 tiles).  The setter rejects anything
// else.
bool w4a4_set_cluster_ctas(int ctas);
int w4a4_get_cluster_ctas();

// The block-scaled FP4 MMA rate (fp4_rate.cu): up to max_pairs CTA pairs,
// one per two SMs, each issuing iters x 4 MMAs of 256 x 256 x 64; cycles[p]
// receives pair p's clock cycles; *pairs how many ran.
cudaError_t launch_fp4_mma_rate(int iters, unsigned long long* cycles, int max_pairs, int* pairs,
                                unsigned int* status, cudaStream_t stream);

// One thread waits on an mbarrier nothing completes; when the bounded wait
// gives up it sets the timeout bit of `status` (selftest.cu).
cudaError_t launch_wait_timeout_selftest(unsigned int* status, cudaStream_t stream);

}  // namespace nvfp4
