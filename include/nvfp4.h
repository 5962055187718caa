/*
 * nvfp4.h -- C ABI of the GB300 (sm_103a) NVFP4 linear-layer library.
 *
 * The method: linear-layer weights are stored as NVFP4 (FP4 E2M1 codes, half a
 * byte per element, plus an FP8 scale per block) and quantised with the
 * FourOverSix rule, which lets every block pick between the usual M=6 scale
 * and an M=4 scale of about 1.5x; GEMMs run as W4A16 (bf16 activations times
 * dequantised weights) for small token counts and as W4A4 (activations
 * quantised online, native block-scaled FP4 tensor-core MMA) above a
 * crossover in M.  Sources: "SOAR 2026 Recap: From Compute Limits to the
 * Open-Source Ecosystem", section "1. Quantization and GEMM dispatch";
 * "SOAR Weekly Champion Notes 07 ... NVFP4 Quantization Improvements",
 * sections "01 Background" and "02 FourOverSix".
 *
 * Formats (readings where the pages are silent; fixed by this library):
 *   - W is [N, K] row-major bf16 (an nn.Linear weight, out x in); X is [M, K]
 *     row-major bf16; Y is [M, N] row-major (bf16, or fp32 when requested).
 *   - Blocks are 16 consecutive elements along K.  codes are [rows, K/2]
 *     bytes, element 2j in the low nibble of byte j and 2j+1 in the high
 *     nibble; code = sign << 3 | E2M1 magnitude bits.
 *   - Block scales are E4M3 bytes.  "Logical" scales are [rows, K/16]
 *     row-major.  "MMA" scales use the block-scaled tensor-core tiling: the
 *     [rows, K/16] matrix is cut into 128 x 4 tiles (zero padded), tiles are
 *     stored row-tile-major, 512 bytes each, with scale (r, c) of a tile at
 *     byte (r % 32) * 16 + (r / 32) * 4 + c.  Size: nvfp4_scales_mma_bytes().
 *   - One FP32 tensor scale ts = amax(|W|) / divisor (divisor 6 * 448 by
 *     default; an all-zero tensor gets ts = 1).  A dequantised element is
 *     value(code) * value(scale) * ts.
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the
 *     library never allocates or frees device memory.  Scratch goes through
 *     the caller's `workspace` (size from nvfp4_workspace_bytes()).
 *   - Every call is asynchronous on `stream`.  Argument errors are returned
 *     synchronously, before anything is launched.  A launch failure returns
 *     NVFP4_ERR_CUDA (text in nvfp4_last_error()).  Errors found on the
 *     device (a non-finite input) are recorded in a device status word and
 *     reported by nvfp4_get_device_status().
 *   - Pointers to tensors must be 16-byte aligned (NVFP4_ERR_ALIGN).
 *   - The library keeps no state between calls except the crossover table
 *     (nvfp4_set_crossover), the W4A16 kernel knob
 *     (nvfp4_set_w4a16_rf_max_m, nvfp4_set_w4a16_sk_max_m), the W4A4 kernel
 *     knob (nvfp4_set_w4a4_cluster), the quantiser launch form
 *     (nvfp4_set_single_launch_quantizer), the activation FourOverSix flag
 *     (nvfp4_set_act_fos), the weight-prefetch flag
 *     (nvfp4_set_weight_prefetch) and the device status word, besides
 *     host-side lookups made once (the driver's tensor-map encoder, per-kernel
 *     occupancy, per-device attributes) and the static scratch array of
 *     nvfp4_linear_noalloc.  Tensor maps are encoded on every call.
 */
#ifndef NVFP4_H_
#define NVFP4_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum nvfp4_status {
  NVFP4_OK = 0,
  NVFP4_ERR_INVALID_ARG = 1, /* null pointer where one is required, bad enum */
  NVFP4_ERR_SHAPE = 2,       /* sizes <= 0 where not allowed, K not a multiple of 16 (64 for the FP4 MMA) */
  NVFP4_ERR_ALIGN = 3,       /* a tensor pointer not 16-byte aligned */
  NVFP4_ERR_WORKSPACE = 4,   /* workspace too small */
  NVFP4_ERR_NONFINITE = 5,   /* an input held Inf or NaN (device-detected) */
  NVFP4_ERR_TIMEOUT = 6,     /* a bounded device-side wait ran out (device-detected) */
  NVFP4_ERR_CUDA = 7,        /* a CUDA runtime or driver call failed */
  NVFP4_ERR_UNSUPPORTED = 8  /* the current GPU is not an sm_103 (GB300), or a size the kernels do not handle */
} nvfp4_status;

/* Output element type of the GEMMs. */
typedef enum nvfp4_out_dtype { NVFP4_OUT_BF16 = 0, NVFP4_OUT_F32 = 1 } nvfp4_out_dtype;

/* Operation ids for nvfp4_workspace_bytes(). */
typedef enum nvfp4_op {
  NVFP4_OP_QUANTIZE_FOS = 0,
  NVFP4_OP_QUANTIZE_ACT = 1,
  NVFP4_OP_GEMM_W4A16 = 2,
  NVFP4_OP_GEMM_W4A4 = 3,
  NVFP4_OP_LINEAR = 4,
  NVFP4_OP_LINEAR_SILU_MUL = 5,
  NVFP4_OP_QAT_BACKWARD = 6,
  NVFP4_OP_GPTQ_FOS = 7
} nvfp4_op;

#define NVFP4_DEFAULT_DIVISOR 2688.0f /* 6 (E2M1 max) * 448 (E4M3 max) */

/* A quantised weight as the GEMMs read it.  All pointers are device pointers,
 * owned by the caller and 16-byte aligned. */
typedef struct nvfp4_weight {
  const uint8_t* codes;      /* [N, K/2] packed E2M1 codes */
  const uint8_t* scales_mma; /* nvfp4_scales_mma_bytes(N, K) bytes, MMA tiling */
  const float* tensor_scale; /* one float */
  int64_t N;
  int64_t K;
} nvfp4_weight;

/* Bytes of an MMA-tiled scale matrix for `rows` rows of length K
 * (= ceil(rows/128) * ceil(K/64) * 512).  Returns 0 for invalid sizes. */
size_t nvfp4_scales_mma_bytes(int64_t rows, int64_t K);

/* Workspace bytes that `op` needs for the given sizes (M is ignored by the
 * quantiser of weights, N by the activation quantiser).  0 on bad sizes. */
size_t nvfp4_workspace_bytes(int op, int64_t M, int64_t N, int64_t K);

/*
 * FourOverSix NVFP4 weight quantisation ("SOAR Weekly Champion Notes 07",
 * section "02 FourOverSix"; round-to-nearest only).
 *
 * For each 16-element block: s6 = E4M3((amax_block / 6) / ts),
 * s4 = E4M3(value(s6) * 1.5); each candidate quantises the block with
 * q = E2M1(x / (value(s) * ts)) and scores it by the binary32 sum of squared
 * dequantisation errors in a fixed order: d = x - value(q) * value(s) * ts
 * rounded once, a_j = d_j^2 + d_(j+8)^2 with one rounding after the second
 * square, then b_j = a_j + a_(j+4), c_j = b_j + b_(j+2), SSE = c_0 + c_1; the
 * block keeps s4 only if its SSE is strictly smaller.  Every step is IEEE
 * binary32, round to nearest even, with no other fused or reordered
 * operation; E4M3 and E2M1 conversions saturate (448, 6).
 *
 *   W            in:  device bf16 [N, K]
 *   N, K         N >= 1, K >= 16, K % 16 == 0
 *   divisor      tensor-scale divisor; <= 0 or non-finite selects 6 * 448
 *   codes        out: device [N, K/2]                          (required)
 *   scales       out: device [N, K/16] logical E4M3 bytes       (nullable)
 *   scales_mma   out: device, nvfp4_scales_mma_bytes(N, K) bytes (nullable;
 *                     padding bytes are written as 0)
 *   tensor_scale out: device, 1 float                          (required)
 *   choice       out: device [N, K/16], 1 = block took M=4      (nullable)
 *   m4_count     out: device, number of M=4 blocks (overwritten) (nullable)
 *   workspace    device scratch of nvfp4_workspace_bytes(NVFP4_OP_QUANTIZE_FOS, 0, N, K)
 * At least one of scales / scales_mma must be given.  On a non-finite input
 * the device status word records NVFP4_ERR_NONFINITE and no output is written.
 */
nvfp4_status nvfp4_quantize_fos(const void* W, int64_t N, int64_t K, float divisor,
                                uint8_t* codes, uint8_t* scales, uint8_t* scales_mma,
                                float* tensor_scale, uint8_t* choice,
                                unsigned long long* m4_count, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream);

/*
 * GPTQ inside FourOverSix scales ("SOAR Weekly Champion Notes 07 ... NVFP4
 * Quantization Improvements", section "03 How we integrated it": each
 * block's M=4 / M=6 choice is fixed first, then GPTQ's error-compensating
 * quantisation runs within it).  Scales, tensor scale (and scales_mma) are
 * those of nvfp4_quantize_fos on W; the codes are GPTQ's: columns quantised
 * in order with those fixed scales, each column's error divided by U[j][j]
 * and spread over the columns not yet quantised along row j of U, the upper
 * Cholesky factor of (H + d I)^-1, d = damp * mean(diag H), in blocks of 128
 * columns.  Every step is binary32 in a fixed order (stated in
 * csrc/gptq.cu), so the codes are reproducible bit for bit.
 *   W        in:  device bf16 [N, K], K <= 11616 (the triangular inverse
 *                 keeps 5 vectors of K floats in shared memory)
 *   H        in:  device fp32 [K, K], symmetric positive semi-definite (the
 *                 layer's Hessian, e.g. 2 X^T X / T over calibration tokens)
 *   damp     in:  >= 0 (GPTQ's usual 0.01)
 *   codes, scales (nullable), scales_mma (nullable), tensor_scale: as
 *                 nvfp4_quantize_fos
 *   workspace nvfp4_workspace_bytes(NVFP4_OP_GPTQ_FOS, 0, N, K) bytes
 * A damped Hessian that is not positive definite sets NVFP4_ERR_NONFINITE in
 * the device status word (nvfp4_get_device_status).  An offline step: about
 * 2K kernel launches for the factorisation.
 */
nvfp4_status nvfp4_gptq_fos(const void* W, int64_t N, int64_t K, const float* H, float damp,
                            uint8_t* codes, uint8_t* scales, uint8_t* scales_mma,
                            float* tensor_scale, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream);

/*
 * Online NVFP4 quantisation of activations for the W4A4 path (the pages give
 * no activation rule; this library uses the standard M=6 scale only, with the
 * same binary32 steps and tensor scale as the weight quantiser).
 *
 *   X            in:  device bf16 [M, K], M >= 1, K >= 16, K % 16 == 0
 *   divisor      tensor-scale divisor; <= 0 or non-finite selects 6 * 448
 *   codes        out: device [M, K/2]                           (required)
 *   scales       out: device [M, K/16] logical                  (nullable)
 *   scales_mma   out: device, nvfp4_scales_mma_bytes(M, K) bytes (nullable)
 *   tensor_scale out: device, 1 float                           (required)
 *   workspace    device scratch of nvfp4_workspace_bytes(NVFP4_OP_QUANTIZE_ACT, M, 0, K)
 * At least one of scales / scales_mma must be given.  A non-finite input is
 * recorded as in nvfp4_quantize_fos.
 */
nvfp4_status nvfp4_quantize_act(const void* X, int64_t M, int64_t K, float divisor,
                                uint8_t* codes, uint8_t* scales, uint8_t* scales_mma,
                                float* tensor_scale, void* workspace, size_t workspace_bytes,
                                cudaStream_t stream);

/*
 * W4A16 GEMM ("SOAR 2026 Recap", section "1. Quantization and GEMM dispatch":
 * the path for M <= 48 on the pages' GPU):
 *   Y[m, n] = ts * sum_k X[m, k] * value(code[n, k]) * value(scale[n, k/16]),
 * bf16 activations, weights dequantised exactly (value(code) * value(scale)
 * has at most 6 significant bits), fp32 accumulation.
 *   X      in:  device bf16 [M, K];  M >= 0 (M == 0 launches nothing)
 *   W      in:  quantised weight; K % 16 == 0
 *   Y      out: device [M, N] of out_dtype
 * For K % 64 != 0 a plain kernel runs (a warp per weight row and 8 tokens,
 * exact binary32 dequantisation, fp32 fma accumulation per lane, a shuffle
 * tree across lanes): the tensor-core kernels stream 64-wide chunks whose
 * rows the TMA can only describe when K % 32 == 0.  For K % 64 == 0 three
 * tensor-core kernels implement it.  For small M (see
 * nvfp4_set_w4a16_sk_max_m): a persistent split-K kernel (one CTA per SM; clusters of up to 8 CTAs each
 * own a run of 128-row weight tiles, CTA r of a cluster a K slice of every
 * one, the slices of a tile summed through distributed shared memory) that
 * keeps its K slice of X in shared memory as f16 scaled per token by a power
 * of two and multiplies exactly dequantised f16 weights with warp-level MMAs.
 * For M <= nvfp4_get_w4a16_rf_max_m(): one CTA per tile and K slice, bf16
 * warp-level MMAs, the slices summed across a cluster.  Above that, weights
 * dequantised into tensor memory for tcgen05 MMAs.  All give the same result
 * up to fp32 summation order, except that the split-K kernel's f16 copy of X
 * rounds elements more than 2^29 below their token's largest magnitude in a
 * K slice (an absolute error below 2^-40 of that magnitude).  The workspace
 * arguments are unused (NULL, 0).
 */
nvfp4_status nvfp4_gemm_w4a16(const void* X, int64_t M, const nvfp4_weight* W, void* Y,
                              int out_dtype, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream);

/*
 * W4A4 GEMM (same section: above the crossover the GEMM runs on the native
 * NVFP4 tensor-core instruction): block-scaled FP4 x FP4 tensor-core MMA with
 * fp32 accumulation,
 *   Y[m, n] = ts_a * ts_w * sum_k value(qa[m,k]) value(sa[m,k/16]) value(qw[n,k]) value(sw[n,k/16]).
 *   a_codes      in: device [M, K/2] (from nvfp4_quantize_act)
 *   a_scales_mma in: device, nvfp4_scales_mma_bytes(M, K) bytes
 *   a_tensor_scale in: device, 1 float
 *   M            >= 0 (M == 0 launches nothing)
 *   W            in: quantised weight; K % 64 == 0 (the MMA's K step;
 *                NVFP4_ERR_SHAPE otherwise)
 *   Y            out: device [M, N] of out_dtype
 * Above 128 tokens the kernel runs on CTA pairs (nvfp4_set_w4a4_cluster).
 * NVFP4_ERR_UNSUPPORTED if no kernel configuration fits the size.  The
 * workspace arguments are unused (NULL, 0).
 */
nvfp4_status nvfp4_gemm_w4a4(const uint8_t* a_codes, const uint8_t* a_scales_mma,
                             const float* a_tensor_scale, int64_t M, const nvfp4_weight* W,
                             void* Y, int out_dtype, void* workspace, size_t workspace_bytes,
                             cudaStream_t stream);

/*
 * NVFP4 linear layer with M-based dispatch (same section: small token counts
 * take W4A16, larger ones W4A4, the two latency curves crossing near M = 48
 * on the pages' GPU, and the faster path is chosen per call).  M <=
 * crossover(N, K), K < 256 or K % 64 != 0 runs nvfp4_gemm_w4a16; otherwise
 * nvfp4_quantize_act (into the workspace) then nvfp4_gemm_w4a4 -- or, with
 * nvfp4_set_act_fos(1), the FourOverSix quantiser on the activations.
 *   workspace  nvfp4_workspace_bytes(NVFP4_OP_LINEAR, M, N, K) bytes
 */
nvfp4_status nvfp4_linear(const void* X, int64_t M, const nvfp4_weight* W, void* Y,
                          int out_dtype, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream);

/*
 * Gated MLP input projection.  "SOAR 2026 Recap ...", section "2. Hybrid
 * attention backend optimization" (GLA linear attention, kernel fusion),
 * fuses an output gate's elementwise work into one kernel with the values
 * kept in registers; this call applies that idea to the MLP's gate: W is the concatenated
 * gate/up weight [2F, K] (rows [0, F) gate, [F, 2F) up), and
 *   Y[m, f] = silu(G[m, f]) * U[m, f],  silu(g) = g / (1 + e^-g),
 * with G = X W_gate^T and U = X W_up^T computed as nvfp4_linear would (same
 * dispatch by M over the whole [2F, K] weight), in binary32.
 *   X          in:  device bf16 [M, K]
 *   W          in:  quantised [2F, K] weight (N = 2F even)
 *   Y          out: device [M, F] of out_dtype
 *   workspace  nvfp4_workspace_bytes(NVFP4_OP_LINEAR_SILU_MUL, M, 2F, K) bytes
 * On the W4A4 branch with bf16 output and F % 128 == 0 the W4A4 kernel
 * applies silu(G) * U in its epilogue: a tile covers 128 features, its 256
 * weight rows the 128 gate rows and the matching up rows (split over the two
 * CTAs of a pair above 128 tokens, in one CTA otherwise), so G and U never
 * reach memory.  Otherwise the GEMM writes fp32 [rows, 2F] into the
 * workspace, 1024 rows at a time, and a separate kernel applies it; the fused
 * and separate forms evaluate the same binary32 expression.
 */
nvfp4_status nvfp4_linear_silu_mul(const void* X, int64_t M, const nvfp4_weight* W, void* Y,
                                   int out_dtype, void* workspace, size_t workspace_bytes,
                                   cudaStream_t stream);

/*
 * NVFP4 -> bf16: out[r, k] = bf16(binary32(value(code) * value(scale) * ts)),
 * the product value(code) * value(scale) exact, one binary32 rounding for the
 * tensor scale, then round to nearest even bf16.
 *   codes [rows, K/2], scales_mma (MMA tiling), tensor_scale (1 float): device
 *   rows >= 0 (0 launches nothing), K >= 16, K % 16 == 0
 *   out   device bf16 [rows, K]
 * Pointers 16-byte aligned (the tensor scale 4-byte).  No workspace.
 */
nvfp4_status nvfp4_dequantize(const uint8_t* codes, const uint8_t* scales_mma,
                              const float* tensor_scale, int64_t rows, int64_t K, void* out,
                              cudaStream_t stream);

/*
 * Backward pass of the FP4-forward linear layer Y = X_hat W_hat^T for
 * quantisation-aware training ("SOAR 2026 Recap ...", section "3. EAGLE-3
 * speculative decoding and hybrid architecture adaptation", paragraph
 * "NVFP4 QAT": the forward GEMM runs in FP4, nvfp4_gemm_w4a4 here, and the
 * gradients pass straight through the quantisers to bf16 master weights):
 *   dX = dY W_hat     (bf16 [M, K]; skipped if dX is NULL)
 *   dW = dY^T X_hat   (fp32 [N, K]; skipped if dW is NULL)
 * with W_hat, X_hat the nvfp4_dequantize bf16 values of W and of the
 * quantised activations (a_codes, a_scales_mma, a_tensor_scale from
 * nvfp4_quantize_act or nvfp4_quantize_fos), fp32 accumulation.  Both
 * products run on this library's tensor-core kernel (tcgen05 kind::f16 on
 * CTA pairs); W_hat^T, X_hat^T and dY^T are formed in the workspace first
 * (dequantised or transposed straight into that layout).
 *   dY         in: device bf16 [M, N]
 *   workspace  nvfp4_workspace_bytes(NVFP4_OP_QAT_BACKWARD, M, N, K) bytes
 */
nvfp4_status nvfp4_qat_backward(const void* dY, int64_t M, const nvfp4_weight* W,
                                const uint8_t* a_codes, const uint8_t* a_scales_mma,
                                const float* a_tensor_scale, void* dX, void* dW, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream);

/* Size of the scratch array built into the library for nvfp4_linear_noalloc
 * (32 MiB, held on every GPU that loads the library until the process exits). */
#define NVFP4_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * nvfp4_linear without a caller-provided workspace, for callers that cannot
 * allocate device memory: plugins inside a host framework that owns every
 * allocation and hands them only its own tensors, embedded runtimes with no
 * device allocator.  The source pages have no counterpart; this is a
 * convenience of this library.
 *
 * Same arguments and result as nvfp4_linear, minus the workspace.  The W4A4
 * branch keeps its scratch (the online-quantised activations) in a fixed
 * NVFP4_NOALLOC_SCRATCH_BYTES array inside the library; a call whose scratch
 * need (nvfp4_workspace_bytes(NVFP4_OP_LINEAR, M, N, K)) exceeds it returns
 * NVFP4_ERR_WORKSPACE with the sizes in nvfp4_last_error().  Roughly, the W4A4
 * branch needs M * (K/2 + K/16) bytes, so at K = 4096 up to about 14,500 rows
 * fit; the W4A16 branch needs none.  No allocator is called.
 *
 * The branch is chosen once per call (M against the crossover table) and the
 * scratch size is checked for that branch.  The first call on each device
 * that takes the W4A4 branch looks up the array's device address (with that
 * device current) and caches it for the current CUDA context (a context
 * re-created after cudaDeviceReset is looked up again); make that first call
 * before any stream capture.  Calls on the W4A16 branch, M == 0 and argument
 * errors never touch the array.  All calls share the one array and it keeps
 * the previous call's contents (nothing in it needs to start at zero): calls
 * that may overlap on the GPU -- on different streams, or from different
 * threads -- race on it and must be serialised by the caller.
 */
nvfp4_status nvfp4_linear_noalloc(const void* X, int64_t M, const nvfp4_weight* W, void* Y,
                                  int out_dtype, cudaStream_t stream);

/* Crossover table: the largest M that still takes the W4A16 path for a
 * weight of shape [N, K].  N == 0 and K == 0 set the default used for shapes
 * without an entry.  Thread-safe.  The built-in default comes from a sweep on
 * GB300 (see nvfp4_get_crossover(0, 0)). */
nvfp4_status nvfp4_set_crossover(int64_t N, int64_t K, int64_t M_threshold);
int64_t nvfp4_get_crossover(int64_t N, int64_t K);

/* Largest M for which nvfp4_gemm_w4a16 uses its register-file kernel
 * (0 ..= 64; default 64).  A tuning knob: both kernels compute the same
 * product.  Thread-safe; returns NVFP4_ERR_INVALID_ARG outside the range. */
nvfp4_status nvfp4_set_w4a16_rf_max_m(int64_t M);
int64_t nvfp4_get_w4a16_rf_max_m(void);

/* Which M nvfp4_gemm_w4a16 sends to its persistent split-K kernel: M <= the
 * value (0 ..= 64), or, for -1 (the default), by the rule measured on GB300:
 * M <= 8, and M <= 16 / M <= 32 on weights of at least 64 / 128 row tiles of
 * 128.  A tuning knob: every kernel computes the same product.  Thread-safe;
 * returns NVFP4_ERR_INVALID_ARG outside -1 ..= 64. */
nvfp4_status nvfp4_set_w4a16_sk_max_m(int64_t M);
int64_t nvfp4_get_w4a16_sk_max_m(void);

/* Weight prefetch (default off).  When on, the W4A16 kernels start reading
 * the weight codes and scales before the previous kernel in the stream has
 * finished (programmatic dependent launch), hiding the HBM latency behind it;
 * the activations are still read, and the output written, only after it.
 * Turn it on only when no work queued on the stream before a GEMM call can
 * still be writing that call's weight buffers -- true when weights are
 * quantised once and then only read, as in inference.  Thread-safe. */
nvfp4_status nvfp4_set_weight_prefetch(int enable);
int nvfp4_get_weight_prefetch(void);

/* FourOverSix for activations (default off).  The pages apply the M=4 / M=6
 * choice to weights and say nothing of activations; when on, nvfp4_linear's
 * W4A4 branch quantises X with the same FourOverSix rule and kernel as
 * nvfp4_quantize_fos (per 16-block: scale 6 or its 1.5x rounding, whichever
 * gives the smaller block squared error; tensor scale amax / 2688) instead of
 * the scale-6-only rule of nvfp4_quantize_act.  nvfp4_quantize_fos itself
 * accepts any bf16 [rows, K] tensor, activations included, and its codes,
 * MMA scales and tensor scale feed nvfp4_gemm_w4a4 as the A operand.
 * Thread-safe. */
nvfp4_status nvfp4_set_act_fos(int enable);
int nvfp4_get_act_fos(void);

/* Quantiser launch form (default off).  On: nvfp4_quantize_fos,
 * nvfp4_quantize_act and the W4A4 branch of the linear calls run one
 * cooperative launch per tensor -- every CTA reads its tiles once, keeping
 * them in shared memory (up to 96 KB per CTA; the rest is read again, from
 * L2 when it fits), a grid-wide barrier forms the tensor amax, then the
 * tiles are quantised.  Off: two launches (an amax pass, then the
 * quantisation pass reading the tensor again).  Both give identical bits;
 * where no cooperative grid can be formed the two-launch form runs.  On GB300
 * the two-launch form measured faster (the arithmetic dominates, and two
 * launches overlap reads with it), hence the default.  Thread-safe. */
nvfp4_status nvfp4_set_single_launch_quantizer(int enable);
int nvfp4_get_single_launch_quantizer(void);

/* W4A4 kernel for M > 128: CTAs per thread-block cluster (default 2).
 *   2: a pair of CTAs shares each 256 x 256 output tile through cta_group::2
 *      MMAs (each CTA stages half of the A rows and half of the B rows of
 *      every K stage, each with its own loads);
 *   1: one CTA per 128 x 256 tile.
 * Where a pair cannot be resident single CTAs are used.  All compute the same product with the same fp32 accumulation
 * order per output.  A tuning knob; thread-safe; NVFP4_ERR_INVALID_ARG for
 * any other value. */
nvfp4_status nvfp4_set_w4a4_cluster(int ctas);
int nvfp4_get_w4a4_cluster(void);

/* Synchronises `stream`, then returns and clears the device status word of the
 * current device: NVFP4_OK, NVFP4_ERR_NONFINITE or NVFP4_ERR_TIMEOUT. */
nvfp4_status nvfp4_get_device_status(cudaStream_t stream);

/*
 * The dense block-scaled FP4 tensor-core rate of this GPU, measured with this
 * library's own instruction stream and no memory traffic: the denominator of
 * the W4A4 roofline fraction (the pages give no FP4 rate; "SOAR 2026 Recap
 * ...", section "1. Quantization and GEMM dispatch", names the NVFP4 MMA as
 * the W4A4 engine).  Launches up to max_pairs CTA pairs (one CTA per SM);
 * each pair issues iters x 4 tcgen05.mma.cta_group::2.kind::mxf4nvf4 of
 * 256 x 256 x 64 (2 * 256 * 256 * 64 flops each) back to back.
 *   iters      1 ..= 2^24
 *   cycles     out: device array of max_pairs; cycles[p] = SM clock cycles
 *              pair p spent issuing and completing its MMAs
 *   pairs      out (host): how many pairs were launched (set before return)
 * Asynchronous on `stream`: time it with events on that stream; flops =
 * pairs * iters * 4 * 2 * 256 * 256 * 64.  NVFP4_ERR_INVALID_ARG for bad
 * arguments, NVFP4_ERR_UNSUPPORTED if no pair fits.
 */
nvfp4_status nvfp4_measure_fp4_mma(int iters, unsigned long long* cycles, int max_pairs, int* pairs,
                                    cudaStream_t stream);

/* Self-test of the bounded device-side wait (the failure path of every
 * pipeline wait in the GEMM kernels): launches one thread that waits on an
 * mbarrier nothing completes.  The wait gives up after its cycle limit (about
 * 1.5 s at 2 GHz) and records NVFP4_ERR_TIMEOUT in the device status word, which
 * the next nvfp4_get_device_status() returns; the CUDA context stays usable.
 * Returns NVFP4_OK once launched. */
nvfp4_status nvfp4_selftest_wait_timeout(cudaStream_t stream);

/* Static text for a status code. */
const char* nvfp4_status_string(nvfp4_status status);

/* Text of the last NVFP4_ERR_CUDA / argument error on this thread. */
const char* nvfp4_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_H_ */
