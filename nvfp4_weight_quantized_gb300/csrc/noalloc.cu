// noalloc.cu -- nvfp4_linear_noalloc: the dispatching linear layer for callers
// that cannot allocate device memory.
//
// nvfp4_linear needs scratch for its W4A4 branch (the activations quantised
// online: codes, MMA-tiled scales, tensor scale and the amax partials).  Some
// callers have no way to provide it: code running while a CUDA graph is being
// captured (where cudaMalloc is not allowed), plugins living inside a host
// framework that owns every allocation, or embedded runtimes without a device
// allocator.  This entry point keeps that scratch in a fixed array that is
// part of the library's device image instead, so it calls no allocator at
// all.  The array (NVFP4_NOALLOC_SCRATCH_BYTES) exists on every GPU that
// loads the library until the process exits.
#include <cstdio>
#include <mutex>

#include "kernels.h"
#include "nvfp4.h"

// The shared scratch.  Its name is only a host-side stand-in: host code must
// use the device address obtained with cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[NVFP4_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and cached.
nvfp4_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (err != cudaSuccess || p == nullptr) return NVFP4_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return NVFP4_OK;
}

}  // namespace

extern "C" nvfp4_status nvfp4_linear_noalloc(const void* X, int64_t M, const nvfp4_weight* W, void* Y,
                                             int out_dtype, cudaStream_t stream) {
  if (W == nullptr) return nvfp4_linear(X, M, W, Y, out_dtype, nullptr, 0, stream);  // reports the error
  // M <= crossover takes the W4A16 branch, which needs no scratch at all;
  // invalid shapes are left to nvfp4_linear to report
  const bool shape_ok = W->N > 0 && W->K >= 256 && W->K % 64 == 0 && M > 0;
  const bool needs_scratch = shape_ok && M > nvfp4_get_crossover(W->N, W->K);
  // the W4A16 branch ignores the workspace, M == 0 launches nothing and bad
  // arguments are reported before any device call: none of them needs the
  // scratch, so none of them looks up its address
  if (!needs_scratch) return nvfp4_linear(X, M, W, Y, out_dtype, nullptr, 0, stream);
  const size_t need = nvfp4_workspace_bytes(NVFP4_OP_LINEAR, M, W->N, W->K);
  if (need == 0 || need > NVFP4_NOALLOC_SCRATCH_BYTES) {
    char msg[160];
    snprintf(msg, sizeof msg,
             "nvfp4_linear_noalloc: M=%lld, K=%lld needs %zu scratch bytes, more than the built-in %u",
             (long long)M, (long long)W->K, need, (unsigned)NVFP4_NOALLOC_SCRATCH_BYTES);
    nvfp4::set_last_error(msg);
    return NVFP4_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  const nvfp4_status st = scratch_address(&scratch);
  if (st != NVFP4_OK) {
    nvfp4::set_last_error("nvfp4_linear_noalloc: cannot look up the scratch address on this device");
    return st;
  }
  return nvfp4_linear(X, M, W, Y, out_dtype, scratch, NVFP4_NOALLOC_SCRATCH_BYTES, stream);
}
