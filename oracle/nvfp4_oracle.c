/*
 * nvfp4_oracle.c -- plain, slow CPU oracle for the NVFP4 linear-layer path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or call this file: only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header, table or
 * constant with the CUDA library; every value below is derived from the
 * format definitions written out in this file.
 *
 * Sources (the method is described on web pages about the SOAR 2026
 * inference contest):
 *   [P1] "SOAR 2026 Recap: From Compute Limits to the Open-Source Ecosystem",
 *        section "1. Quantization and GEMM dispatch": linear weights are
 *        stored as NVFP4 (FP4 E2M1, half a byte per element); each block
 *        picks between scale=4 and scale=6; GEMMs run W4A16 for M <= 48 and
 *        W4A4 (native NVFP4 MMA) above.
 *   [P3] "SOAR Weekly Champion Notes 07 ... NVFP4 Quantization Improvements",
 *        section "01 Background": the E2M1 value set {0, +-0.5, +-1, +-1.5,
 *        +-2, +-3, +-4, +-6}, maximum 6, standard blocks normalised to
 *        [-6, 6] (M=6);
 *        section "02 FourOverSix": the M=4 scale is the M=6 scale times 1.5,
 *        re-rounded to FP8; each block keeps the scale whose block mean
 *        squared dequantisation error is smaller (strictly smaller for M=4);
 *        the output stays standard NVFP4 (4-bit codes + FP8 block scale).
 *
 * Where the pages are silent this file takes the following readings (the
 * CUDA path takes the same ones):
 *   - 16-element blocks along K, E4M3 block scales, one FP32 tensor scale
 *     ts = amax(|W|) / D with D = 6 * 448 by default; an all-zero tensor
 *     gets ts = 1.
 *   - Every step of the quantiser is IEEE binary32 with round-to-nearest-even;
 *     the only fused multiply-adds are the explicit fmaf calls (build with
 *     -ffp-contract=off so the compiler adds none):
 *       r6  = (amax_block / 6) / ts,      s6 = E4M3(r6)
 *       s4  = E4M3(value(s6) * 1.5)
 *       eff = value(s) * ts
 *       q_i = E2M1(x_i / eff)   (q_i = signed zero when eff == 0)
 *       d_i = x_i - value(q_i) * eff        rounded once (exact product)
 *       a_j = d_j * d_j + RN(d_j+8 * d_j+8)  rounded once, j < 8
 *       b_j = a_j + a_j+4,  c_j = b_j + b_j+2,  SSE = c_0 + c_1
 *     and the block keeps s4 iff SSE4 < SSE6 (ties keep M=6).  Comparing
 *     sums is the same as comparing means: division by 16 is exact.  The
 *     error and the first level of the square-sum are single-rounding
 *     (fused) operations: the pages fix no precision or order for the block
 *     MSE, and this form is the more exact one.
 *   - E4M3 and E2M1 conversions round to nearest, ties to the even code, and
 *     saturate to the largest finite value (448 and 6).  The sign of a code
 *     is the sign of x (so negative values that round to zero give -0).
 *   - Code packing: element 2j in the low nibble of byte j, 2j+1 in the high.
 *   - Activations (W4A4 path) use the standard M=6 rule only.
 *   - GEMM reference: the plain definition, sum_k x[m,k] * w_hat[n,k] in
 *     binary64, with w_hat = value(code) * value(scale) * ts (exact).
 *
 * parity pinned: see the test suite (format tables against a third-party
 * library, worked examples computed by hand, brute-force scale search,
 * invariants; the GEMMs against a library matmul; the bf16 dequantisation
 * by exact cases and hand-worked ties; GPTQ by the identity-Hessian case, its
 * inverse factor against a library inverse and the least-squares
 * continuation of every row).
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_ERR_SHAPE 2
#define OR_ERR_NONFINITE 5
#define DEFAULT_DIVISOR_F 2688.0f /* 6 * 448 */

/* ------------------------------------------------------------------------ */
/* Formats                                                                  */
/* ------------------------------------------------------------------------ */

/* bfloat16: the upper 16 bits of an IEEE binary32. */
float oracle_bf16_value(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* FP4 E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit, no
 * infinities or NaN.  Exponent field 0 is subnormal: 0.m * 2^0. */
double oracle_e2m1_value(uint8_t code) {
  int s = (code >> 3) & 1;
  int e = (code >> 1) & 3;
  int m = code & 1;
  double mag = (e == 0) ? (m * 0.5) : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

/* FP8 E4M3 (the "fn" variant): 1 sign, 4 exponent bits (bias 7), 3 mantissa
 * bits; exponent field 0 is subnormal (0.mmm * 2^-6); S.1111.111 is NaN and
 * there is no infinity, so the largest finite magnitude is 1.75 * 2^8 = 448. */
double oracle_e4m3_value(uint8_t byte) {
  int s = (byte >> 7) & 1;
  int e = (byte >> 3) & 15;
  int m = byte & 7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) mag = ldexp(m / 8.0, -6);
  else mag = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -mag : mag;
}

/* Round |v| to the nearest E2M1 magnitude (ties to the even code), saturate
 * at 6, and attach the sign of v.  Written as a search over the 8
 * magnitudes so that it reads as the definition of rounding to nearest. */
uint8_t oracle_e2m1_encode(float v) {
  uint8_t sign = signbit(v) ? 8 : 0;
  double a = fabs((double)v);
  if (a >= 6.0) return sign | 7; /* also catches +inf */
  int best = 0;
  double best_d = a;
  for (int m = 1; m < 8; ++m) {
    double d = fabs(a - oracle_e2m1_value((uint8_t)m));
    if (d < best_d || (d == best_d && (m & 1) == 0)) {
      best = m;
      best_d = d;
    }
  }
  return sign | (uint8_t)best;
}

/* Round |v| to the nearest finite E4M3 magnitude (ties to the even code),
 * saturating at 448, sign from v.  Search over the 127 finite magnitudes. */
uint8_t oracle_e4m3_encode(float v) {
  uint8_t sign = signbit(v) ? 0x80 : 0;
  double a = fabs((double)v);
  if (a >= 448.0) return sign | 0x7E;
  int best = 0;
  double best_d = a;
  for (int c = 1; c < 127; ++c) {
    double d = fabs(a - oracle_e4m3_value((uint8_t)c));
    if (d < best_d || (d == best_d && (c & 1) == 0)) {
      best = c;
      best_d = d;
    }
  }
  return sign | (uint8_t)best;
}

/* ------------------------------------------------------------------------ */
/* One 16-element block, quantised with a given scale byte.                 */
/* ------------------------------------------------------------------------ */

/* Quantise 16 values with block scale byte s and tensor scale ts; return the
 * block's sum of squared dequantisation errors in the fixed binary32 order
 * described at the top of this file.  q receives one code per element. */
float oracle_block_sse(const float x[16], uint8_t s, float ts, uint8_t q[16]) {
  float eff = (float)oracle_e4m3_value(s) * ts;
  float d[16];
  for (int i = 0; i < 16; ++i) {
    if (eff == 0.0f) {
      q[i] = signbit(x[i]) ? 8 : 0;
      d[i] = x[i];
    } else {
      float r = x[i] / eff;
      q[i] = oracle_e2m1_encode(r);
      /* x - value * eff with one rounding (value * eff is exact in double,
       * and fmaf rounds the exact result once) */
      d[i] = fmaf(-(float)oracle_e2m1_value(q[i]), eff, x[i]);
    }
  }
  float a[8], b[4], c[2];
  for (int j = 0; j < 8; ++j) a[j] = fmaf(d[j], d[j], d[j + 8] * d[j + 8]);
  for (int j = 0; j < 4; ++j) b[j] = a[j] + a[j + 4];
  for (int j = 0; j < 2; ++j) c[j] = b[j] + b[j + 2];
  return c[0] + c[1];
}

/* The standard (M=6) scale of a block: E4M3((amax_block / 6) / ts). */
uint8_t oracle_block_scale_m6(const float x[16], float ts) {
  float amax = 0.0f;
  for (int i = 0; i < 16; ++i) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  float r6 = (amax / 6.0f) / ts;
  return oracle_e4m3_encode(r6);
}

/* FourOverSix on one block.  Outputs: q (chosen codes), the chosen scale byte,
 * the choice (1 = M4), and both candidates' scale bytes and SSEs. */
void oracle_fos_block(const float x[16], float ts, uint8_t q[16], uint8_t* scale,
                      uint8_t* choice, uint8_t* s6_out, uint8_t* s4_out,
                      float* sse6_out, float* sse4_out) {
  uint8_t s6 = oracle_block_scale_m6(x, ts);
  float s6v = (float)oracle_e4m3_value(s6);
  uint8_t s4 = oracle_e4m3_encode(s6v * 1.5f);
  uint8_t q6[16], q4[16];
  float sse6 = oracle_block_sse(x, s6, ts, q6);
  float sse4 = oracle_block_sse(x, s4, ts, q4);
  int m4 = sse4 < sse6;
  memcpy(q, m4 ? q4 : q6, 16);
  *scale = m4 ? s4 : s6;
  *choice = (uint8_t)m4;
  if (s6_out) *s6_out = s6;
  if (s4_out) *s4_out = s4;
  if (sse6_out) *sse6_out = sse6;
  if (sse4_out) *sse4_out = sse4;
}

/* ------------------------------------------------------------------------ */
/* Whole tensors                                                             */
/* ------------------------------------------------------------------------ */

/* Tensor scale: amax(|X|) / divisor, or 1 for an all-zero tensor.  Returns
 * OR_ERR_NONFINITE if any element is Inf or NaN. */
int oracle_tensor_scale(const uint16_t* X, int64_t count, float divisor, float* ts) {
  float amax = 0.0f;
  for (int64_t i = 0; i < count; ++i) {
    float v = oracle_bf16_value(X[i]);
    if (!isfinite(v)) return OR_ERR_NONFINITE;
    float a = fabsf(v);
    if (a > amax) amax = a;
  }
  *ts = (amax == 0.0f) ? 1.0f : amax / divisor;
  return OR_OK;
}

static void pack_codes(const uint8_t q[16], uint8_t* out8) {
  for (int j = 0; j < 8; ++j) out8[j] = (uint8_t)((q[2 * j] & 15) | ((q[2 * j + 1] & 15) << 4));
}

/* Quantise rows of a bf16 matrix with a given tensor scale: FourOverSix when
 * fos != 0, otherwise the standard M=6 scale only.  codes [rows, K/2],
 * scales [rows, K/16], choice [rows, K/16] (nullable).  Returns the number of
 * blocks that took M=4. */
uint64_t oracle_quantize_rows(const uint16_t* X, int64_t rows, int64_t K, float ts, int fos,
                              uint8_t* codes, uint8_t* scales, uint8_t* choice) {
  uint64_t count = 0;
  int64_t nb = K / 16;
  for (int64_t n = 0; n < rows; ++n) {
    for (int64_t b = 0; b < nb; ++b) {
      float x[16];
      for (int i = 0; i < 16; ++i) x[i] = oracle_bf16_value(X[n * K + b * 16 + i]);
      uint8_t q[16], s, c = 0;
      if (fos) {
        oracle_fos_block(x, ts, q, &s, &c, NULL, NULL, NULL, NULL);
      } else {
        s = oracle_block_scale_m6(x, ts);
        (void)oracle_block_sse(x, s, ts, q);
      }
      pack_codes(q, codes + n * (K / 2) + b * 8);
      scales[n * nb + b] = s;
      if (choice) choice[n * nb + b] = c;
      count += c;
    }
  }
  return count;
}

/* FourOverSix NVFP4 weight quantisation of W [N, K] (bf16 bits, row-major).
 * codes [N, K/2], scales [N, K/16] (E4M3 bytes, row-major), choice [N, K/16]
 * (nullable, 1 = M4), m4_count (nullable). */
int oracle_quantize_fos(const uint16_t* W, int64_t N, int64_t K, float divisor,
                        uint8_t* codes, uint8_t* scales, uint8_t* choice,
                        float* ts_out, uint64_t* m4_count) {
  if (N <= 0 || K <= 0 || K % 16 != 0) return OR_ERR_SHAPE;
  float ts;
  int st = oracle_tensor_scale(W, N * K, divisor, &ts);
  if (st != OR_OK) return st;
  *ts_out = ts;
  uint64_t count = oracle_quantize_rows(W, N, K, ts, 1, codes, scales, choice);
  if (m4_count) *m4_count = count;
  return OR_OK;
}

/* Standard (M=6 only) NVFP4 quantisation of activations X [M, K]. */
int oracle_quantize_act(const uint16_t* X, int64_t M, int64_t K, float divisor,
                        uint8_t* codes, uint8_t* scales, float* ts_out) {
  if (M <= 0 || K <= 0 || K % 16 != 0) return OR_ERR_SHAPE;
  float ts;
  int st = oracle_tensor_scale(X, M * K, divisor, &ts);
  if (st != OR_OK) return st;
  *ts_out = ts;
  (void)oracle_quantize_rows(X, M, K, ts, 0, codes, scales, NULL);
  return OR_OK;
}

/* Block-scaled tensor-core scale layout.  The scale matrix [R, K/16] is cut
 * into tiles of 128 rows x 4 scale columns (zero-padded at the edges); tiles
 * are stored row-tile-major, each as 512 bytes in which scale (r, c) of the
 * tile sits at byte (r mod 32) * 16 + (r div 32) * 4 + c. */
int64_t oracle_scales_mma_bytes(int64_t R, int64_t K) {
  int64_t rt = (R + 127) / 128;
  int64_t ct = (K / 16 + 3) / 4;
  return rt * ct * 512;
}

void oracle_scales_to_mma(const uint8_t* scales, int64_t R, int64_t K, uint8_t* out) {
  int64_t nb = K / 16;
  int64_t ct = (nb + 3) / 4;
  memset(out, 0, (size_t)oracle_scales_mma_bytes(R, K));
  for (int64_t r = 0; r < R; ++r) {
    for (int64_t c = 0; c < nb; ++c) {
      int64_t tile = (r / 128) * ct + (c / 4);
      int64_t rr = r % 128, cc = c % 4;
      out[tile * 512 + (rr % 32) * 16 + (rr / 32) * 4 + cc] = scales[r * nb + c];
    }
  }
}

/* Dequantised element (n, k) of an NVFP4 matrix, exact in binary64. */
static double dequant(const uint8_t* codes, const uint8_t* scales, float ts, int64_t K,
                      int64_t n, int64_t k) {
  uint8_t byte = codes[n * (K / 2) + k / 2];
  uint8_t code = (k & 1) ? (byte >> 4) : (byte & 15);
  return oracle_e2m1_value(code) * oracle_e4m3_value(scales[n * (K / 16) + k / 16]) * (double)ts;
}

/* W4A16: Y[m, n] = sum_k X[m, k] * w_hat[n, k] in binary64. */
int oracle_gemm_w4a16(const uint16_t* X, int64_t M, int64_t K, const uint8_t* codes,
                      const uint8_t* scales, float ts, int64_t N, double* Y) {
  if (M < 0 || N <= 0 || K <= 0 || K % 16 != 0) return OR_ERR_SHAPE;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k)
        acc += (double)oracle_bf16_value(X[m * K + k]) * dequant(codes, scales, ts, K, n, k);
      Y[m * N + n] = acc;
    }
  return OR_OK;
}

/* Rows `rows[0..R)` of the W4A16 product only (for sampled checks). */
int oracle_gemm_w4a16_rows(const uint16_t* X, const int64_t* rows, int64_t R, int64_t K,
                           const uint8_t* codes, const uint8_t* scales, float ts, int64_t N,
                           double* Y) {
  for (int64_t i = 0; i < R; ++i) {
    int st = oracle_gemm_w4a16(X + rows[i] * K, 1, K, codes, scales, ts, N, Y + i * N);
    if (st != OR_OK) return st;
  }
  return OR_OK;
}

/* W4A4: Y[m, n] = sum_k x_hat[m, k] * w_hat[n, k] in binary64. */
int oracle_gemm_w4a4(const uint8_t* a_codes, const uint8_t* a_scales, float a_ts, int64_t M,
                     const uint8_t* w_codes, const uint8_t* w_scales, float w_ts, int64_t N,
                     int64_t K, double* Y) {
  if (M < 0 || N <= 0 || K <= 0 || K % 16 != 0) return OR_ERR_SHAPE;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k)
        acc += dequant(a_codes, a_scales, a_ts, K, m, k) * dequant(w_codes, w_scales, w_ts, K, n, k);
      Y[m * N + n] = acc;
    }
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Dequantisation to bf16 (the operand of the QAT backward GEMMs)            */
/* ------------------------------------------------------------------------ */

/* Round a finite binary32 to bfloat16, to nearest, ties to the even bit
 * pattern: the 16 dropped bits are compared with half of the last kept bit. */
static uint16_t bf16_round(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  uint32_t kept = u >> 16, dropped = u & 0xFFFFu;
  if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))) kept += 1u;
  return (uint16_t)kept;
}

/* "SOAR 2026 Recap ...", section "3. EAGLE-3 speculative decoding and hybrid
 * architecture adaptation", paragraph "NVFP4 QAT": the draft's forward GEMM
 * runs in FP4 and its gradients go straight through to bf16 master weights,
 * so the backward GEMMs take bf16 operands.  Reading: its NVFP4 operand is taken to
 * bf16 in two steps, value(code) * value(scale) (exact: at most 2 + 4
 * significant bits) times the tensor scale rounded once to binary32, then
 * rounded to bfloat16.  codes [R, K/2], scales logical [R, K/16]. */
int oracle_dequant_bf16(const uint8_t* codes, const uint8_t* scales, float ts, int64_t R, int64_t K,
                        uint16_t* out) {
  if (R < 0 || K <= 0 || K % 16 != 0) return OR_ERR_SHAPE;
  for (int64_t r = 0; r < R; ++r)
    for (int64_t k = 0; k < K; ++k) {
      uint8_t byte = codes[r * (K / 2) + k / 2];
      uint8_t code = (k & 1) ? (byte >> 4) : (byte & 15);
      float vs = (float)(oracle_e2m1_value(code) * oracle_e4m3_value(scales[r * (K / 16) + k / 16]));
      float q = vs * ts; /* binary32, one rounding */
      out[r * K + k] = bf16_round(q);
    }
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* GPTQ with FourOverSix scales                                             */
/* ------------------------------------------------------------------------ */

/* "SOAR Weekly Champion Notes 07 ... NVFP4 Quantization Improvements",
 * section "03 How we integrated it": FourOverSix first fixes each block's
 * scale (M=4 or M=6), then GPTQ quantises inside that choice.  GPTQ itself (the method the pages
 * combine it with) quantises the columns of W in order and spreads each
 * column's error, divided by the diagonal of U, over the columns still to be
 * quantised through the rows of U, the upper Cholesky factor of the inverse
 * of the damped Hessian (H + d I, d = damp * mean(diag H)), in blocks of
 * `block` columns: inside a block the error goes to the block's remaining
 * columns at once, to the columns after the block once per block.
 *
 * Every step below is binary32 with one rounding per operation, in the order
 * written (the kernel's precision: the codes are decided in binary32):
 *   d      = damp * ((sum_k H[k][k], k ascending) / K)
 *   A      = J (H + d I) J, J the index reversal
 *   L      = chol(A), right-looking: for j: L[j][j] = sqrt(A[j][j]),
 *            L[i][j] = A[i][j] / L[j][j], then A[i][c] = fma(-L[i][j], L[c][j], A[i][c])
 *            for j < c <= i
 *   Linv   = L^-1 by columns: x[j] = 1 / L[j][j]; for i > j:
 *            s = sum_{k=j}^{i-1} fma(L[i][k], x[k], s) (k ascending), x[i] = -s / L[i][i]
 *   U      = J Linv J  (then H'^-1 = U^T U)
 *   column j of row n, block scale eff = value(scale) * ts:
 *            q = e2m1(RN(w / eff)) (q = sign only when eff == 0),
 *            e = fma(-value(q), eff, w) / U[j][j],
 *            w[n][c] = fma(-e, U[j][c], w[n][c]) for the block's later columns c,
 *   after a block, for every later column c:
 *            s = sum_{j in block} fma(E[n][j], U[j][c], s) (j ascending), w[n][c] -= s.
 * Scales and ts are those of oracle_quantize_fos on the original W.  H is
 * [K, K] row-major (symmetric); U_out (nullable) receives U [K, K].
 * Returns OR_ERR_NONFINITE if a Cholesky pivot is not positive. */
int oracle_gptq_fos(const uint16_t* W, int64_t N, int64_t K, const float* H, float damp, int64_t block,
                    uint8_t* codes, uint8_t* scales, float* ts_out, float* U_out) {
  if (N <= 0 || K <= 0 || K % 16 != 0 || block <= 0 || block % 16 != 0) return OR_ERR_SHAPE;
  int st = oracle_quantize_fos(W, N, K, DEFAULT_DIVISOR_F, codes, scales, NULL, ts_out, NULL);
  if (st != OR_OK) return st;
  const float ts = *ts_out;
  float* A = (float*)malloc(sizeof(float) * K * K);
  float* Li = (float*)malloc(sizeof(float) * K * K);
  float* Wc = (float*)malloc(sizeof(float) * N * K);
  float* E = (float*)malloc(sizeof(float) * N * block);
  if (!A || !Li || !Wc || !E) {
    free(A); free(Li); free(Wc); free(E);
    return OR_ERR_SHAPE;
  }
  float dsum = 0.0f;
  for (int64_t k = 0; k < K; ++k) dsum += H[k * K + k];
  const float dval = damp * (dsum / (float)K);
  for (int64_t i = 0; i < K; ++i)
    for (int64_t j = 0; j < K; ++j) {
      float h = H[(K - 1 - i) * K + (K - 1 - j)];
      A[i * K + j] = (i == j) ? h + dval : h;
    }
  /* Cholesky, lower triangle of A in place */
  for (int64_t j = 0; j < K && st == OR_OK; ++j) {
    if (!(A[j * K + j] > 0.0f)) {
      st = OR_ERR_NONFINITE;
      break;
    }
    const float p = sqrtf(A[j * K + j]);
    A[j * K + j] = p;
    for (int64_t i = j + 1; i < K; ++i) A[i * K + j] = A[i * K + j] / p;
    for (int64_t i = j + 1; i < K; ++i)
      for (int64_t c = j + 1; c <= i; ++c) A[i * K + c] = fmaf(-A[i * K + j], A[c * K + j], A[i * K + c]);
  }
  if (st == OR_OK) {
    /* inverse of the lower factor, column by column */
    memset(Li, 0, sizeof(float) * K * K);
    for (int64_t j = 0; j < K; ++j) {
      Li[j * K + j] = 1.0f / A[j * K + j];
      for (int64_t i = j + 1; i < K; ++i) {
        float s = 0.0f;
        for (int64_t k = j; k < i; ++k) s = fmaf(A[i * K + k], Li[k * K + j], s);
        Li[i * K + j] = -s / A[i * K + i];
      }
    }
#define U_AT(i, j) Li[(K - 1 - (i)) * K + (K - 1 - (j))]
    if (U_out)
      for (int64_t i = 0; i < K; ++i)
        for (int64_t j = 0; j < K; ++j) U_out[i * K + j] = U_AT(i, j);
    for (int64_t i = 0; i < N * K; ++i) Wc[i] = oracle_bf16_value(W[i]);
    const int64_t nb = K / 16;
    for (int64_t b0 = 0; b0 < K; b0 += block) {
      const int64_t b1 = b0 + block < K ? b0 + block : K;
      for (int64_t n = 0; n < N; ++n) {
        float* w = Wc + n * K;
        for (int64_t j = b0; j < b1; ++j) {
          const float eff = (float)oracle_e4m3_value(scales[n * nb + j / 16]) * ts;
          uint8_t q;
          float d;
          if (eff == 0.0f) {
            q = signbit(w[j]) ? 8 : 0;
            d = w[j];
          } else {
            q = oracle_e2m1_encode(w[j] / eff);
            d = fmaf(-(float)oracle_e2m1_value(q), eff, w[j]);
          }
          const float e = d / U_AT(j, j);
          E[n * block + (j - b0)] = e;
          for (int64_t c = j + 1; c < b1; ++c) w[c] = fmaf(-e, U_AT(j, c), w[c]);
          uint8_t* byte = codes + n * (K / 2) + j / 2;
          *byte = (j & 1) ? (uint8_t)((*byte & 15) | (q << 4)) : (uint8_t)((*byte & 0xF0) | q);
        }
        for (int64_t c = b1; c < K; ++c) {
          float s = 0.0f;
          for (int64_t j = b0; j < b1; ++j) s = fmaf(E[n * block + (j - b0)], U_AT(j, c), s);
          w[c] = w[c] - s;
        }
      }
    }
#undef U_AT
  }
  free(A);
  free(Li);
  free(Wc);
  free(E);
  return st;
}

/* ------------------------------------------------------------------------ */
/* GPTQ with FourOverSix scales, plain binary64 form                        */
/* ------------------------------------------------------------------------ */

/* Lower Cholesky factor of the symmetric positive definite A [K, K] (binary64,
 * textbook column form), in place in the lower triangle; 0 on success. */
static int chol64(double* A, int64_t K) {
  for (int64_t j = 0; j < K; ++j) {
    double d = A[j * K + j];
    for (int64_t k = 0; k < j; ++k) d -= A[j * K + k] * A[j * K + k];
    if (!(d > 0.0)) return -1;
    d = sqrt(d);
    A[j * K + j] = d;
    for (int64_t i = j + 1; i < K; ++i) {
      double s = A[i * K + j];
      for (int64_t k = 0; k < j; ++k) s -= A[i * K + k] * A[j * K + k];
      A[i * K + j] = s / d;
    }
  }
  return 0;
}

/* The same GPTQ as oracle_gptq_fos, written from its definition with none of
 * that function's binary32 order: every quantity in binary64, no blocking.
 *   Hd    = H + d I, d = damp * mean(diag H);
 *   Hinv  = Hd^-1 (Cholesky of Hd, then its inverse);
 *   U     = the upper-triangular factor with Hinv = U^T U (Cholesky of Hinv,
 *           transposed);
 *   for each row, columns j in order: q = nearest E2M1 value of w[j] / eff
 *   (ties to even, saturating at 6; eff = value(scale) * ts of the given
 *   FourOverSix scales), e = (w[j] - value(q) eff) / U[j][j], and every later
 *   column c gets w[c] -= e U[j][c] at once.
 * follow (nullable): the codes of another GPTQ run over the same W, H and
 * scales.  Where this run's |w[j] / eff| lies within `delta` of an E2M1
 * rounding midpoint the followed code is taken instead (so both runs go on
 * from the same decision), near[n * K + j] is set to 1, and the followed
 * value must be one of the two grid values either side of that midpoint
 * (else OR_ERR_SHAPE).  codes receives the decisions (sign of zero from the
 * quotient).  OR_ERR_NONFINITE if Hd or Hinv is not positive definite. */
int oracle_gptq_fos_ref64(const uint16_t* W, int64_t N, int64_t K, const float* H, double damp,
                          const uint8_t* scales, float ts, const uint8_t* follow, double delta, uint8_t* codes,
                          uint8_t* near) {
  static const double grid[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  if (N <= 0 || K <= 0 || K % 16 != 0) return OR_ERR_SHAPE;
  double* A = (double*)malloc(sizeof(double) * K * K);
  double* Inv = (double*)malloc(sizeof(double) * K * K);
  double* w = (double*)malloc(sizeof(double) * K);
  if (!A || !Inv || !w) {
    free(A); free(Inv); free(w);
    return OR_ERR_SHAPE;
  }
  int st = OR_OK;
  double dsum = 0.0;
  for (int64_t k = 0; k < K; ++k) dsum += (double)H[k * K + k];
  const double dval = damp * (dsum / (double)K);
  for (int64_t i = 0; i < K * K; ++i) A[i] = (double)H[i];
  for (int64_t k = 0; k < K; ++k) A[k * K + k] += dval;
  if (chol64(A, K) != 0) st = OR_ERR_NONFINITE;
  if (st == OR_OK) {
    /* Hd^-1 = L^-T L^-1: solve L Y = I column by column, then L^T Z = Y */
    for (int64_t c = 0; c < K; ++c) {
      for (int64_t i = 0; i < K; ++i) { /* forward */
        double s = (i == c) ? 1.0 : 0.0;
        for (int64_t k = 0; k < i; ++k) s -= A[i * K + k] * Inv[k * K + c];
        Inv[i * K + c] = s / A[i * K + i];
      }
      for (int64_t i = K - 1; i >= 0; --i) { /* backward */
        double s = Inv[i * K + c];
        for (int64_t k = i + 1; k < K; ++k) s -= A[k * K + i] * Inv[k * K + c];
        Inv[i * K + c] = s / A[i * K + i];
      }
    }
    /* symmetrise (the two triangles agree up to rounding), then factor */
    for (int64_t i = 0; i < K; ++i)
      for (int64_t j = 0; j < i; ++j) {
        const double v = 0.5 * (Inv[i * K + j] + Inv[j * K + i]);
        Inv[i * K + j] = Inv[j * K + i] = v;
      }
    if (chol64(Inv, K) != 0) st = OR_ERR_NONFINITE; /* lower C, Hinv = C C^T, U = C^T */
  }
#define U64(i, j) Inv[(j) * K + (i)]
  for (int64_t n = 0; n < N && st == OR_OK; ++n) {
    for (int64_t k = 0; k < K; ++k) w[k] = (double)oracle_bf16_value(W[n * K + k]);
    for (int64_t j = 0; j < K && st == OR_OK; ++j) {
      const double eff = oracle_e4m3_value(scales[n * (K / 16) + j / 16]) * (double)ts;
      uint8_t q, nflag = 0;
      double d;
      if (eff == 0.0) {
        q = signbit(w[j]) ? 8 : 0;
        d = w[j];
      } else {
        const double x = w[j] / eff, ax = fabs(x);
        int best = 0;
        for (int g = 1; g < 8; ++g) {
          const double dg = fabs(ax - grid[g]), db = fabs(ax - grid[best]);
          if (dg < db || (dg == db && (g & 1) == 0)) best = g; /* ties to the even code */
        }
        /* distance to the nearest rounding midpoint */
        double md = 1e300;
        for (int g = 0; g < 7; ++g) {
          const double m = fabs(ax - 0.5 * (grid[g] + grid[g + 1]));
          if (m < md) md = m;
        }
        q = (uint8_t)((x < 0.0 || (x == 0.0 && signbit(x)) ? 8 : 0) | best);
        if (follow != NULL && md < delta) {
          const uint8_t byte = follow[n * (K / 2) + j / 2];
          const uint8_t fq = (j & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
          const int fm = fq & 7;
          /* the midpoint next to ax, and the grid values either side of it */
          int lo = 0;
          for (int g = 0; g < 7; ++g)
            if (fabs(ax - 0.5 * (grid[g] + grid[g + 1])) == md) lo = g;
          if (fm != lo && fm != lo + 1) st = OR_ERR_SHAPE;
          if (fm != 0 && ((fq & 8) != 0) != (x < 0.0)) st = OR_ERR_SHAPE;
          q = fq;
          nflag = 1;
        }
        d = w[j] - grid[q & 7] * ((q & 8) ? -1.0 : 1.0) * eff;
      }
      if (near != NULL) near[n * K + j] = nflag;
      const double e = d / U64(j, j);
      for (int64_t c = j + 1; c < K; ++c) w[c] -= e * U64(j, c);
      uint8_t* byte = codes + n * (K / 2) + j / 2;
      *byte = (j & 1) ? (uint8_t)((*byte & 15) | (q << 4)) : (uint8_t)((*byte & 0xF0) | q);
    }
  }
#undef U64
  free(A);
  free(Inv);
  free(w);
  return st;
}
