// api.cu -- the C ABI (include/nvfp4.h): argument checks, workspace layout,
// dispatch between the W4A16 and W4A4 paths, device status word.
#include <cuda.h>

#include <cmath>
#include <atomic>
#include <cstdio>
#include <map>
#include <mutex>
#include <string>
#include <utility>

#include "common.cuh"
#include "kernels.h"
#include "nvfp4.h"

// Device status word of this library (one per device): bit 0 = non-finite
// input seen, bit 1 = a bounded wait ran out.
static __device__ unsigned int g_device_status;

namespace {

thread_local std::string t_last_error;

std::mutex g_mu;
// Largest M that still takes the W4A16 path, per weight shape (N, K), and for
// shapes without an entry.  Built-in values: the crossover of graph-timed
// W4A16 vs activation quantisation + W4A4 measured on GB300 with
// nvfp4_weight_quantized_gb300.tune (sweep M = 1..256, cold weights, weight
// prefetch on); re-run it to retune.
std::map<std::pair<int64_t, int64_t>, int64_t> g_crossover = {
    {{4096, 4096}, 64}, {{11008, 4096}, 16}, {{22016, 4096}, 8}, {{4096, 11008}, 64}};
int64_t g_default_crossover = 48;
// Largest M that nvfp4_gemm_w4a16 sends to the register-file kernel.
std::atomic<int64_t> g_w4a16_rf_max_m{64};
// Largest M that nvfp4_gemm_w4a16 sends to the persistent split-K kernel, or
// -1: by the measured rule in nvfp4_gemm_w4a16.
std::atomic<int64_t> g_w4a16_sk_max_m{-1};
// Whether GEMM kernels may read the weights before the previous kernel in the
// stream has finished (nvfp4_set_weight_prefetch).
std::atomic<bool> g_weight_prefetch{false};
// Whether nvfp4_linear's W4A4 branch quantises activations with FourOverSix
// (nvfp4_set_act_fos) instead of the M=6 scale only.
std::atomic<bool> g_act_fos{false};

struct DeviceInfo {
  bool ready = false;
  unsigned long long ctx_id = 0;  // the context the addresses below belong to
  int num_sms = 0;
  unsigned int* status = nullptr;
};
constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];

nvfp4_status fail(nvfp4_status st, const char* what) {
  t_last_error = what;
  return st;
}

nvfp4_status fail_cuda(cudaError_t err, const char* where) {
  t_last_error = std::string(where) + ": " + cudaGetErrorString(err);
  return NVFP4_ERR_CUDA;
}

// Per-device set-up, done with that device current, once per CUDA context
// on it (a context re-created after cudaDeviceReset loads the library's
// device image again, at possibly different addresses): SM count, a check
// that this is an sm_103 GPU, and the device address of the status word.
nvfp4_status device_info(const DeviceInfo** out) {
  int dev = -1;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return fail_cuda(err, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(NVFP4_ERR_UNSUPPORTED, "device index out of range");
  unsigned long long ctx = 0;
  if (!nvfp4::current_context_id(&ctx)) return fail(NVFP4_ERR_CUDA, "cannot identify the current CUDA context");
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready || d.ctx_id != ctx) {
    d.ready = false;
    int major = 0, minor = 0;
    err = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return fail_cuda(err, "cudaDeviceGetAttribute");
    if (major != 10 || minor != 3)
      return fail(NVFP4_ERR_UNSUPPORTED, "this library is built for sm_103a (GB300) only");
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_device_status);
    if (err != cudaSuccess) return fail_cuda(err, "cudaGetSymbolAddress(status)");
    d.status = static_cast<unsigned int*>(p);
    d.ctx_id = ctx;
    d.ready = true;
  }
  *out = &d;
  return NVFP4_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

float effective_divisor(float d) { return (d > 0.0f && std::isfinite(d)) ? d : NVFP4_DEFAULT_DIVISOR; }

constexpr int64_t kMaxElems = int64_t(1) << 40;

bool weight_ok(const nvfp4_weight* W) {
  return W != nullptr && W->codes != nullptr && W->scales_mma != nullptr && W->tensor_scale != nullptr;
}

// A weight descriptor: K a multiple of 16 (one NVFP4 block); the FP4 tensor-core
// paths (W4A4, and the QAT forward it serves) need K % 64 == 0 as well.
nvfp4_status check_weight(const nvfp4_weight* W, int k_multiple = 16) {
  if (!weight_ok(W)) return fail(NVFP4_ERR_INVALID_ARG, "weight descriptor or one of its pointers is null");
  if (W->N <= 0 || W->K <= 0 || W->K % 16 != 0 || W->N > kMaxElems / W->K)
    return fail(NVFP4_ERR_SHAPE, "weight needs N >= 1, K >= 16, K % 16 == 0");
  if (W->K % k_multiple != 0)
    return fail(NVFP4_ERR_SHAPE, "the FP4 tensor-core path needs K % 64 == 0");
  if (!aligned(W->codes, 16) || !aligned(W->scales_mma, 16) || !aligned(W->tensor_scale, 4))
    return fail(NVFP4_ERR_ALIGN, "weight pointers must be 16-byte aligned");
  return NVFP4_OK;
}

nvfp4_status check_out_dtype(int out_dtype) {
  if (out_dtype != NVFP4_OUT_BF16 && out_dtype != NVFP4_OUT_F32)
    return fail(NVFP4_ERR_INVALID_ARG, "out_dtype must be NVFP4_OUT_BF16 or NVFP4_OUT_F32");
  return NVFP4_OK;
}

nvfp4_status quantize_common(const void* X, int64_t rows, int64_t K, float divisor, bool fos, uint8_t* codes,
                             uint8_t* scales, uint8_t* scales_mma, float* ts, uint8_t* choice,
                             unsigned long long* m4_count, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (X == nullptr || codes == nullptr || ts == nullptr || (scales == nullptr && scales_mma == nullptr))
    return fail(NVFP4_ERR_INVALID_ARG, "X, codes, tensor_scale and one of scales/scales_mma are required");
  if (rows <= 0 || K < 16 || K % 16 != 0 || rows > kMaxElems / K)
    return fail(NVFP4_ERR_SHAPE, "need rows >= 1, K >= 16, K % 16 == 0");
  if (!aligned(X, 16) || !aligned(codes, 16) || !aligned(scales, 16) || !aligned(scales_mma, 16) ||
      !aligned(choice, 16) || !aligned(ts, 4) || !aligned(m4_count, 8))
    return fail(NVFP4_ERR_ALIGN, "tensor pointers must be 16-byte aligned");
  if (ws == nullptr || ws_bytes < nvfp4::quant_workspace_bytes() || !aligned(ws, 16))
    return fail(NVFP4_ERR_WORKSPACE, "workspace missing, unaligned or too small");
  const DeviceInfo* d = nullptr;
  nvfp4_status st = device_info(&d);
  if (st != NVFP4_OK) return st;
  cudaError_t err = nvfp4::launch_quantize(X, rows, K, effective_divisor(divisor), fos, codes, scales,
                                           scales_mma, ts, choice, m4_count, ws, d->status, d->num_sms, stream);
  if (err != cudaSuccess) return fail_cuda(err, "quantize launch");
  return NVFP4_OK;
}

struct LinearWs {
  size_t codes_off, scales_off, ts_off, quant_off, total;
};

// Rows of the fp32 [rows, 2F] GEMM output that nvfp4_linear_silu_mul stages
// in its workspace when silu(G) * U is not fused into the GEMM (a multiple of
// the 128-row scale tiles, so a chunk's activation scales are contiguous).
constexpr int64_t kSiluChunkRows = 1024;

LinearWs linear_ws_layout(int64_t M, int64_t K) {
  LinearWs l;
  l.codes_off = 0;
  l.scales_off = align256((size_t)M * (size_t)(K / 2));
  l.ts_off = l.scales_off + align256(nvfp4_scales_mma_bytes(M, K));
  l.quant_off = l.ts_off + 256;
  l.total = l.quant_off + align256(nvfp4::quant_workspace_bytes());
  return l;
}

}  // namespace

namespace nvfp4 {
void set_last_error(const char* what) { t_last_error = what; }

bool current_context_id(unsigned long long* id) {
  typedef CUresult (*GetCurrentFn)(CUcontext*);
  typedef CUresult (*GetIdFn)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(p);
  });
  if (get_current == nullptr || get_id == nullptr) return false;
  CUcontext c = nullptr;
  if (get_current(&c) != CUDA_SUCCESS) return false;
  if (c == nullptr) {
    // the runtime has not made its primary context current on this thread
    // yet (a call that binds it; never reached while a stream is captured,
    // since capturing needs the context already)
    if (cudaFree(nullptr) != cudaSuccess || get_current(&c) != CUDA_SUCCESS || c == nullptr) return false;
  }
  return get_id(c, id) == CUDA_SUCCESS;
}
}  // namespace nvfp4

extern "C" {

size_t nvfp4_scales_mma_bytes(int64_t rows, int64_t K) {
  if (rows <= 0 || K <= 0 || K % 16 != 0) return 0;
  return (size_t)((rows + 127) / 128) * (size_t)((K / 16 + 3) / 4) * 512;
}

size_t nvfp4_workspace_bytes(int op, int64_t M, int64_t N, int64_t K) {
  (void)N;
  if (K <= 0 || K % 16 != 0) return 0;
  switch (op) {
    case NVFP4_OP_QUANTIZE_FOS:
    case NVFP4_OP_QUANTIZE_ACT: return nvfp4::quant_workspace_bytes();
    case NVFP4_OP_GEMM_W4A16:
    case NVFP4_OP_GEMM_W4A4: return 0;
    case NVFP4_OP_LINEAR:
      // sized for the W4A4 branch whatever the current crossover is
      if (M <= 0) return 0;
      return linear_ws_layout(M, K).total;
    case NVFP4_OP_GPTQ_FOS:
      // the GPTQ working set, logical scales, the quantiser's partials
      if (N <= 0) return 0;
      return nvfp4::gptq_workspace_bytes(N, K) + align256((size_t)N * (size_t)(K / 16)) +
             align256(nvfp4::quant_workspace_bytes());
    case NVFP4_OP_QAT_BACKWARD:
      // transposed bf16 operands of the two tensor-core GEMMs
      if (M <= 0 || N <= 0) return 0;
      return nvfp4::qat_workspace_bytes(M, N, K);
    case NVFP4_OP_LINEAR_SILU_MUL:
      // the linear workspace, then fp32 [min(M, chunk), N] for an unfused silu(G) * U
      if (M <= 0 || N <= 0) return 0;
      return linear_ws_layout(M, K).total + align256((size_t)std::min(M, kSiluChunkRows) * (size_t)N * 4);
    default: return 0;
  }
}

nvfp4_status nvfp4_quantize_fos(const void* W, int64_t N, int64_t K, float divisor, uint8_t* codes,
                                uint8_t* scales, uint8_t* scales_mma, float* tensor_scale, uint8_t* choice,
                                unsigned long long* m4_count, void* workspace, size_t workspace_bytes,
                                cudaStream_t stream) {
  return quantize_common(W, N, K, divisor, true, codes, scales, scales_mma, tensor_scale, choice, m4_count,
                         workspace, workspace_bytes, stream);
}

nvfp4_status nvfp4_quantize_act(const void* X, int64_t M, int64_t K, float divisor, uint8_t* codes,
                                uint8_t* scales, uint8_t* scales_mma, float* tensor_scale, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream) {
  return quantize_common(X, M, K, divisor, false, codes, scales, scales_mma, tensor_scale, nullptr, nullptr,
                         workspace, workspace_bytes, stream);
}

nvfp4_status nvfp4_gemm_w4a16(const void* X, int64_t M, const nvfp4_weight* W, void* Y, int out_dtype,
                              void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  (void)workspace;
  (void)workspace_bytes;
  nvfp4_status st = check_weight(W);
  if (st != NVFP4_OK) return st;
  if ((st = check_out_dtype(out_dtype)) != NVFP4_OK) return st;
  if (M < 0 || M > kMaxElems / W->K || M > kMaxElems / W->N) return fail(NVFP4_ERR_SHAPE, "bad M");
  if (M == 0) return NVFP4_OK;
  if (X == nullptr || Y == nullptr) return fail(NVFP4_ERR_INVALID_ARG, "X and Y are required");
  if (!aligned(X, 16) || !aligned(Y, 16)) return fail(NVFP4_ERR_ALIGN, "X and Y must be 16-byte aligned");
  const DeviceInfo* d = nullptr;
  if ((st = device_info(&d)) != NVFP4_OK) return st;
  const bool f32 = out_dtype == NVFP4_OUT_F32, pf = g_weight_prefetch.load(std::memory_order_relaxed);
  if (W->K % 64 != 0) {  // rows the 64-wide tensor-core kernels cannot stream
    const cudaError_t e = nvfp4::launch_gemm_w4a16_any(X, M, W->codes, W->scales_mma, W->tensor_scale, W->N, W->K,
                                                       Y, f32, d->num_sms, stream);
    if (e != cudaSuccess) return fail_cuda(e, "gemm_w4a16 launch");
    return NVFP4_OK;
  }
  const int64_t sk_max = g_w4a16_sk_max_m.load(std::memory_order_relaxed);
  const int64_t rf_max = g_w4a16_rf_max_m.load(std::memory_order_relaxed);
  cudaError_t err = cudaErrorNotSupported;
  // by default split-K up to 8 tokens, and up to 16 / 32 on weights of at
  // least 64 / 128 row tiles, where it measured faster than the cluster split
  // kernel on GB300
  const int64_t tiles = (W->N + 127) / 128;
  const bool sk = sk_max < 0 ? (M <= 8 || (M <= 16 && tiles >= 64) || (M <= 32 && tiles >= 128)) : M <= sk_max;
  if (sk)
    err = nvfp4::launch_gemm_w4a16_sk(X, M, W->codes, W->scales_mma, W->tensor_scale, W->N, W->K, Y, f32, pf,
                                      d->status, d->num_sms, stream);
  if (err == cudaErrorNotSupported) {
    // the split-K kernel declines shapes whose activation slice does not fit
    // in shared memory: the cluster split kernel takes those
    if (M <= rf_max || sk)
      err = nvfp4::launch_gemm_w4a16_rf(X, M, W->codes, W->scales_mma, W->tensor_scale, W->N, W->K, Y, f32, pf,
                                        d->status, d->num_sms, stream);
    else
      err = nvfp4::launch_gemm_w4a16(X, M, W->codes, W->scales_mma, W->tensor_scale, W->N, W->K, Y, f32,
                                     d->status, d->num_sms, stream);
  }
  if (err == cudaErrorNotSupported) return fail(NVFP4_ERR_UNSUPPORTED, "gemm_w4a16: unsupported size");
  if (err != cudaSuccess) return fail_cuda(err, "gemm_w4a16 launch");
  return NVFP4_OK;
}

nvfp4_status nvfp4_gemm_w4a4(const uint8_t* a_codes, const uint8_t* a_scales_mma, const float* a_tensor_scale,
                             int64_t M, const nvfp4_weight* W, void* Y, int out_dtype, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
  (void)workspace;
  (void)workspace_bytes;
  nvfp4_status st = check_weight(W, 64);
  if (st != NVFP4_OK) return st;
  if ((st = check_out_dtype(out_dtype)) != NVFP4_OK) return st;
  if (M < 0 || M > kMaxElems / W->K || M > kMaxElems / W->N) return fail(NVFP4_ERR_SHAPE, "bad M");
  if (M == 0) return NVFP4_OK;
  if (a_codes == nullptr || a_scales_mma == nullptr || a_tensor_scale == nullptr || Y == nullptr)
    return fail(NVFP4_ERR_INVALID_ARG, "activation codes, scales, tensor scale and Y are required");
  if (!aligned(a_codes, 16) || !aligned(a_scales_mma, 16) || !aligned(a_tensor_scale, 4) || !aligned(Y, 16))
    return fail(NVFP4_ERR_ALIGN, "activation and output pointers must be 16-byte aligned");
  const DeviceInfo* d = nullptr;
  if ((st = device_info(&d)) != NVFP4_OK) return st;
  cudaError_t err = nvfp4::launch_gemm_w4a4(a_codes, a_scales_mma, a_tensor_scale, M, W->codes, W->scales_mma,
                                            W->tensor_scale, W->N, W->K, Y, out_dtype == NVFP4_OUT_F32,
                                            d->status, d->num_sms, stream);
  if (err == cudaErrorNotSupported) return fail(NVFP4_ERR_UNSUPPORTED, "gemm_w4a4: unsupported size");
  if (err != cudaSuccess) return fail_cuda(err, "gemm_w4a4 launch");
  return NVFP4_OK;
}

nvfp4_status nvfp4_linear(const void* X, int64_t M, const nvfp4_weight* W, void* Y, int out_dtype,
                          void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  nvfp4_status st = check_weight(W);
  if (st != NVFP4_OK) return st;
  return nvfp4::linear_branch(X, M, W, Y, out_dtype, workspace, workspace_bytes, stream,
                              nvfp4::linear_takes_w4a4(M, W->N, W->K));
}

}  // extern "C"

namespace nvfp4 {

bool linear_takes_w4a4(int64_t M, int64_t N, int64_t K) {
  // the tensor-core path needs at least one full 256-wide K stage and K % 64 == 0
  return !(M <= nvfp4_get_crossover(N, K) || K < 256 || K % 64 != 0);
}

nvfp4_status linear_branch(const void* X, int64_t M, const nvfp4_weight* W, void* Y, int out_dtype,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream, bool w4a4) {
  nvfp4_status st = check_weight(W);
  if (st != NVFP4_OK) return st;
  if (!w4a4 || W->K < 256 || W->K % 64 != 0)
    return nvfp4_gemm_w4a16(X, M, W, Y, out_dtype, workspace, workspace_bytes, stream);
  if ((st = check_out_dtype(out_dtype)) != NVFP4_OK) return st;
  if (M > kMaxElems / W->K) return fail(NVFP4_ERR_SHAPE, "bad M");
  const LinearWs l = linear_ws_layout(M, W->K);
  if (workspace == nullptr || workspace_bytes < l.total || !aligned(workspace, 256))
    return fail(NVFP4_ERR_WORKSPACE, "linear: workspace missing, not 256-byte aligned or too small");
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* a_codes = ws + l.codes_off;
  uint8_t* a_smma = ws + l.scales_off;
  float* a_ts = reinterpret_cast<float*>(ws + l.ts_off);
  st = quantize_common(X, M, W->K, NVFP4_DEFAULT_DIVISOR, g_act_fos.load(std::memory_order_relaxed), a_codes,
                       nullptr, a_smma, a_ts, nullptr, nullptr, ws + l.quant_off, workspace_bytes - l.quant_off,
                       stream);
  if (st != NVFP4_OK) return st;
  return nvfp4_gemm_w4a4(a_codes, a_smma, a_ts, M, W, Y, out_dtype, nullptr, 0, stream);
}

}  // namespace nvfp4

extern "C" {

nvfp4_status nvfp4_linear_silu_mul(const void* X, int64_t M, const nvfp4_weight* W, void* Y, int out_dtype,
                                   void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  nvfp4_status st = check_weight(W);
  if (st != NVFP4_OK) return st;
  if ((st = check_out_dtype(out_dtype)) != NVFP4_OK) return st;
  if (W->N % 2 != 0) return fail(NVFP4_ERR_SHAPE, "linear_silu_mul: W needs an even number of rows (gate, up)");
  if (M < 0 || M > kMaxElems / W->K || M > kMaxElems / W->N) return fail(NVFP4_ERR_SHAPE, "bad M");
  if (M == 0) return NVFP4_OK;
  if (X == nullptr || Y == nullptr) return fail(NVFP4_ERR_INVALID_ARG, "X and Y are required");
  if (!aligned(X, 16) || !aligned(Y, 16)) return fail(NVFP4_ERR_ALIGN, "X and Y must be 16-byte aligned");
  const int64_t N = W->N, F = N / 2, K = W->K;
  const LinearWs l = linear_ws_layout(M, K);
  const size_t need = nvfp4_workspace_bytes(NVFP4_OP_LINEAR_SILU_MUL, M, N, K);
  if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256))
    return fail(NVFP4_ERR_WORKSPACE, "linear_silu_mul: workspace missing, not 256-byte aligned or too small");
  const DeviceInfo* d = nullptr;
  if ((st = device_info(&d)) != NVFP4_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* y2 = reinterpret_cast<float*>(ws + l.total);  // fp32 [chunk, 2F]
  const bool f32 = out_dtype == NVFP4_OUT_F32;
  const size_t out_elt = f32 ? 4 : 2;
  cudaError_t err;
  if (M <= nvfp4_get_crossover(N, K) || K < 256 || K % 64 != 0) {
    // W4A16 into fp32, then silu(G) * U
    for (int64_t r0 = 0; r0 < M; r0 += kSiluChunkRows) {
      const int64_t mc = std::min(kSiluChunkRows, M - r0);
      st = nvfp4_gemm_w4a16(static_cast<const uint8_t*>(X) + (size_t)r0 * K * 2, mc, W, y2, NVFP4_OUT_F32,
                            nullptr, 0, stream);
      if (st != NVFP4_OK) return st;
      if ((err = nvfp4::launch_silu_mul(y2, mc, F, static_cast<uint8_t*>(Y) + (size_t)r0 * F * out_elt, f32,
                                        stream)) != cudaSuccess)
        return fail_cuda(err, "silu_mul launch");
    }
    return NVFP4_OK;
  }
  uint8_t* a_codes = ws + l.codes_off;
  uint8_t* a_smma = ws + l.scales_off;
  float* a_ts = reinterpret_cast<float*>(ws + l.ts_off);
  st = quantize_common(X, M, K, NVFP4_DEFAULT_DIVISOR, g_act_fos.load(std::memory_order_relaxed), a_codes, nullptr,
                       a_smma, a_ts, nullptr, nullptr, ws + l.quant_off, l.total - l.quant_off, stream);
  if (st != NVFP4_OK) return st;
  if (!f32) {
    // silu(G) * U in the epilogue of the W4A4 kernel (CTA pairs above 128
    // tokens, single CTAs otherwise)
    err = nvfp4::launch_gemm_w4a4_gate_up(a_codes, a_smma, a_ts, M, W->codes, W->scales_mma, W->tensor_scale, N, K,
                                          Y, d->status, d->num_sms, stream);
    if (err == cudaSuccess) return NVFP4_OK;
    if (err != cudaErrorNotSupported) return fail_cuda(err, "gemm_w4a4 gate/up launch");
  }
  const size_t ct = (size_t)((K / 16 + 3) / 4);  // scale column tiles per 128-row tile
  for (int64_t r0 = 0; r0 < M; r0 += kSiluChunkRows) {
    const int64_t mc = std::min(kSiluChunkRows, M - r0);
    st = nvfp4_gemm_w4a4(a_codes + (size_t)r0 * (K / 2), a_smma + (size_t)(r0 / 128) * ct * 512, a_ts, mc, W, y2,
                         NVFP4_OUT_F32, nullptr, 0, stream);
    if (st != NVFP4_OK) return st;
    if ((err = nvfp4::launch_silu_mul(y2, mc, F, static_cast<uint8_t*>(Y) + (size_t)r0 * F * out_elt, f32,
                                      stream)) != cudaSuccess)
      return fail_cuda(err, "silu_mul launch");
  }
  return NVFP4_OK;
}

nvfp4_status nvfp4_gptq_fos(const void* W, int64_t N, int64_t K, const float* H, float damp, uint8_t* codes,
                            uint8_t* scales, uint8_t* scales_mma, float* tensor_scale, void* workspace,
                            size_t workspace_bytes, cudaStream_t stream) {
  if (W == nullptr || H == nullptr || codes == nullptr || tensor_scale == nullptr)
    return fail(NVFP4_ERR_INVALID_ARG, "gptq_fos: W, H, codes and tensor_scale are required");
  if (!(damp >= 0.0f) || !std::isfinite(damp)) return fail(NVFP4_ERR_INVALID_ARG, "gptq_fos: damp must be >= 0");
  if (N <= 0 || K < 16 || K % 16 != 0 || N > kMaxElems / K || K > nvfp4::gptq_max_k())
    return fail(NVFP4_ERR_SHAPE, "gptq_fos: need N >= 1, 16 <= K <= 11616, K % 16 == 0");
  if (!aligned(H, 16)) return fail(NVFP4_ERR_ALIGN, "gptq_fos: H must be 16-byte aligned");
  const size_t gws = nvfp4::gptq_workspace_bytes(N, K), sbytes = align256((size_t)N * (size_t)(K / 16));
  if (workspace == nullptr || !aligned(workspace, 256) ||
      workspace_bytes < nvfp4_workspace_bytes(NVFP4_OP_GPTQ_FOS, 0, N, K))
    return fail(NVFP4_ERR_WORKSPACE, "gptq_fos: workspace missing, not 256-byte aligned or too small");
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* lscales = scales != nullptr ? scales : ws + gws;
  // 1. FourOverSix on the original weights fixes every block's scale (and ts)
  nvfp4_status st = quantize_common(W, N, K, NVFP4_DEFAULT_DIVISOR, true, codes, lscales, scales_mma, tensor_scale,
                                    nullptr, nullptr, ws + gws + sbytes, workspace_bytes - gws - sbytes, stream);
  if (st != NVFP4_OK) return st;
  const DeviceInfo* d = nullptr;
  if ((st = device_info(&d)) != NVFP4_OK) return st;
  // 2. GPTQ inside those scales rewrites the codes
  const cudaError_t err =
      nvfp4::launch_gptq(W, N, K, H, damp, lscales, tensor_scale, codes, workspace, d->status, stream);
  if (err != cudaSuccess) return fail_cuda(err, "gptq launch");
  return NVFP4_OK;
}

nvfp4_status nvfp4_dequantize(const uint8_t* codes, const uint8_t* scales_mma, const float* tensor_scale,
                              int64_t rows, int64_t K, void* out, cudaStream_t stream) {
  if (codes == nullptr || scales_mma == nullptr || tensor_scale == nullptr || out == nullptr)
    return fail(NVFP4_ERR_INVALID_ARG, "dequantize: codes, scales_mma, tensor_scale and out are required");
  if (rows < 0 || K < 16 || K % 16 != 0 || rows > kMaxElems / K)
    return fail(NVFP4_ERR_SHAPE, "dequantize: need rows >= 0, K >= 16, K % 16 == 0");
  if (!aligned(codes, 16) || !aligned(scales_mma, 16) || !aligned(tensor_scale, 4) || !aligned(out, 16))
    return fail(NVFP4_ERR_ALIGN, "dequantize: pointers must be 16-byte aligned");
  if (rows == 0) return NVFP4_OK;
  nvfp4_status st;
  const DeviceInfo* d = nullptr;
  if ((st = device_info(&d)) != NVFP4_OK) return st;
  const cudaError_t err = nvfp4::launch_dequant_bf16(codes, scales_mma, tensor_scale, rows, K, out, d->num_sms, stream);
  if (err != cudaSuccess) return fail_cuda(err, "dequantize launch");
  return NVFP4_OK;
}

nvfp4_status nvfp4_qat_backward(const void* dY, int64_t M, const nvfp4_weight* W, const uint8_t* a_codes,
                                const uint8_t* a_scales_mma, const float* a_tensor_scale, void* dX, void* dW,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  nvfp4_status st = check_weight(W, 64);
  if (st != NVFP4_OK) return st;
  const int64_t N = W->N, K = W->K;
  if (M < 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX || M > kMaxElems / K || M > kMaxElems / N)
    return fail(NVFP4_ERR_SHAPE, "qat_backward: bad M");
  if (M == 0 || (dX == nullptr && dW == nullptr)) return NVFP4_OK;
  if (dY == nullptr || (dW != nullptr && (a_codes == nullptr || a_scales_mma == nullptr || a_tensor_scale == nullptr)))
    return fail(NVFP4_ERR_INVALID_ARG, "qat_backward: dY (and the quantised activations for dW) are required");
  if (!aligned(dY, 16) || (dX != nullptr && !aligned(dX, 16)) || (dW != nullptr && !aligned(dW, 16)))
    return fail(NVFP4_ERR_ALIGN, "qat_backward: pointers must be 16-byte aligned");
  if (workspace == nullptr || !aligned(workspace, 256) ||
      workspace_bytes < nvfp4_workspace_bytes(NVFP4_OP_QAT_BACKWARD, M, N, K))
    return fail(NVFP4_ERR_WORKSPACE, "qat_backward: workspace missing, not 256-byte aligned or too small");
  const DeviceInfo* d = nullptr;
  if ((st = device_info(&d)) != NVFP4_OK) return st;
  const cudaError_t err = nvfp4::qat_backward(dY, M, W->codes, W->scales_mma, W->tensor_scale, N, K, a_codes,
                                              a_scales_mma, a_tensor_scale, dX, dW, workspace, d->status, stream);
  if (err == cudaErrorNotSupported) return fail(NVFP4_ERR_UNSUPPORTED, "qat_backward: unsupported size");
  if (err != cudaSuccess) return fail_cuda(err, "qat_backward launch");
  return NVFP4_OK;
}

nvfp4_status nvfp4_set_crossover(int64_t N, int64_t K, int64_t M_threshold) {
  if (N < 0 || K < 0 || M_threshold < 0) return fail(NVFP4_ERR_INVALID_ARG, "negative crossover argument");
  std::lock_guard<std::mutex> lk(g_mu);
  if (N == 0 && K == 0) g_default_crossover = M_threshold;
  else g_crossover[{N, K}] = M_threshold;
  return NVFP4_OK;
}

nvfp4_status nvfp4_set_w4a16_rf_max_m(int64_t M) {
  if (M < 0 || M > nvfp4::w4a16_rf_max_tokens()) return fail(NVFP4_ERR_INVALID_ARG, "w4a16 rf max M out of range");
  g_w4a16_rf_max_m.store(M, std::memory_order_relaxed);
  return NVFP4_OK;
}

int64_t nvfp4_get_w4a16_rf_max_m(void) { return g_w4a16_rf_max_m.load(std::memory_order_relaxed); }

nvfp4_status nvfp4_set_w4a16_sk_max_m(int64_t M) {
  if (M < -1 || M > nvfp4::w4a16_sk_max_tokens()) return fail(NVFP4_ERR_INVALID_ARG, "w4a16 sk max M out of range");
  g_w4a16_sk_max_m.store(M, std::memory_order_relaxed);
  return NVFP4_OK;
}

int64_t nvfp4_get_w4a16_sk_max_m(void) { return g_w4a16_sk_max_m.load(std::memory_order_relaxed); }

nvfp4_status nvfp4_set_w4a4_cluster(int ctas) {
  if (!nvfp4::w4a4_set_cluster_ctas(ctas)) return fail(NVFP4_ERR_INVALID_ARG, "w4a4 cluster size must be 1 or 2");
  return NVFP4_OK;
}

int nvfp4_get_w4a4_cluster(void) { return nvfp4::w4a4_get_cluster_ctas(); }

nvfp4_status nvfp4_set_weight_prefetch(int enable) {
  g_weight_prefetch.store(enable != 0, std::memory_order_relaxed);
  return NVFP4_OK;
}

int nvfp4_get_weight_prefetch(void) { return g_weight_prefetch.load(std::memory_order_relaxed) ? 1 : 0; }

nvfp4_status nvfp4_set_single_launch_quantizer(int enable) {
  nvfp4::quantize_set_single_launch(enable != 0);
  return NVFP4_OK;
}

int nvfp4_get_single_launch_quantizer(void) { return nvfp4::quantize_get_single_launch() ? 1 : 0; }

nvfp4_status nvfp4_set_act_fos(int enable) {
  g_act_fos.store(enable != 0, std::memory_order_relaxed);
  return NVFP4_OK;
}

int nvfp4_get_act_fos(void) { return g_act_fos.load(std::memory_order_relaxed) ? 1 : 0; }

int64_t nvfp4_get_crossover(int64_t N, int64_t K) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_crossover.find({N, K});
  return it == g_crossover.end() ? g_default_crossover : it->second;
}

nvfp4_status nvfp4_measure_fp4_mma(int iters, unsigned long long* cycles, int max_pairs, int* pairs,
                                    cudaStream_t stream) {
  if (pairs == nullptr || cycles == nullptr || iters <= 0 || iters > (1 << 24) || max_pairs <= 0)
    return fail(NVFP4_ERR_INVALID_ARG, "measure_fp4_mma: need cycles, pairs, 0 < iters <= 2^24, max_pairs > 0");
  *pairs = 0;
  const DeviceInfo* d = nullptr;
  const nvfp4_status st = device_info(&d);
  if (st != NVFP4_OK) return st;
  const cudaError_t err = nvfp4::launch_fp4_mma_rate(iters, cycles, max_pairs, pairs, d->status, stream);
  if (err == cudaErrorNotSupported) return fail(NVFP4_ERR_UNSUPPORTED, "measure_fp4_mma: no CTA pair fits");
  if (err != cudaSuccess) return fail_cuda(err, "measure_fp4_mma launch");
  return NVFP4_OK;
}

nvfp4_status nvfp4_selftest_wait_timeout(cudaStream_t stream) {
  const DeviceInfo* d = nullptr;
  const nvfp4_status st = device_info(&d);
  if (st != NVFP4_OK) return st;
  const cudaError_t err = nvfp4::launch_wait_timeout_selftest(d->status, stream);
  if (err != cudaSuccess) return fail_cuda(err, "wait-timeout self-test launch");
  return NVFP4_OK;
}

nvfp4_status nvfp4_get_device_status(cudaStream_t stream) {
  cudaError_t err = cudaStreamSynchronize(stream);
  if (err != cudaSuccess) return fail_cuda(err, "cudaStreamSynchronize");
  unsigned int v = 0;
  err = cudaMemcpyFromSymbol(&v, g_device_status, sizeof v);
  if (err != cudaSuccess) return fail_cuda(err, "read status word");
  const unsigned int zero = 0;
  err = cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero);
  if (err != cudaSuccess) return fail_cuda(err, "clear status word");
  if (v & nvfp4::kStatusNonfinite) return NVFP4_ERR_NONFINITE;
  if (v & nvfp4::kStatusTimeout) return NVFP4_ERR_TIMEOUT;
  return NVFP4_OK;
}

const char* nvfp4_status_string(nvfp4_status s) {
  switch (s) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_INVALID_ARG: return "invalid argument";
    case NVFP4_ERR_SHAPE: return "unsupported or inconsistent shape";
    case NVFP4_ERR_ALIGN: return "pointer not 16-byte aligned";
    case NVFP4_ERR_WORKSPACE: return "workspace missing or too small";
    case NVFP4_ERR_NONFINITE: return "non-finite input";
    case NVFP4_ERR_TIMEOUT: return "device-side wait timed out";
    case NVFP4_ERR_CUDA: return "CUDA error";
    case NVFP4_ERR_UNSUPPORTED: return "unsupported device or size";
  }
  return "unknown status";
}

const char* nvfp4_last_error(void) { return t_last_error.c_str(); }

}  // extern "C"
