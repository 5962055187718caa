// noalloc.cu -- nvfp4_linear_noalloc: the dispatching linear layer for callers
// that cannot allocate device memory.
//
// nvfp4_linear needs scratch for its W4A4 branch (the activations quantised
// online: codes, MMA-tiled scales, tensor scale and the amax partials).  Some
// callers have no way to provide it: plugins living inside a host framework
// that owns every allocation and hands out only the tensors it manages, or
// embedded runtimes that have no device allocator at all.  This entry point
// keeps that scratch in a fixed array that is part of the library's device
// image instead, so it calls no allocator.  The array
// (NVFP4_NOALLOC_SCRATCH_BYTES) exists on every GPU that loads the library
// until the process exits.
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
struct ScratchAddr {
  unsigned long long ctx_id = 0;  // the context the address belongs to
  void* addr = nullptr;
};
ScratchAddr g_scratch[kMaxDevices];

// Device address of the scratch on the current device, looked up with that
// device current the first time it is needed in each CUDA context (a context
// re-created after cudaDeviceReset loads the array again, possibly at another
// address) and cached.
nvfp4_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_CUDA;
  unsigned long long ctx = 0;
  if (!nvfp4::current_context_id(&ctx)) return NVFP4_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  ScratchAddr& s = g_scratch[dev];
  if (s.addr == nullptr || s.ctx_id != ctx) {
    void* p = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (err != cudaSuccess || p == nullptr) return NVFP4_ERR_CUDA;
    s.addr = p;
    s.ctx_id = ctx;
  }
  *out = s.addr;
  return NVFP4_OK;
}

}  // namespace

extern "C" nvfp4_status nvfp4_linear_noalloc(const void* X, int64_t M, const nvfp4_weight* W, void* Y,
                                             int out_dtype, cudaStream_t stream) {
  if (W == nullptr) return nvfp4_linear(X, M, W, Y, out_dtype, nullptr, 0, stream);  // reports the error
  // The branch is chosen once, here, and passed down, so the scratch size
  // checked below is the one the executed branch uses even if another thread
  // changes the crossover table meanwhile.  Invalid shapes are left to
  // nvfp4_linear's checks to report.
  const bool shape_ok = W->N > 0 && W->K >= 256 && W->K % 64 == 0 && M > 0;
  const bool w4a4 = shape_ok && nvfp4::linear_takes_w4a4(M, W->N, W->K);
  // the W4A16 branch needs no workspace, M == 0 launches nothing and bad
  // arguments are reported before any device call: none of them needs the
  // scratch, so none of them looks up its address
  if (!w4a4) return nvfp4::linear_branch(X, M, W, Y, out_dtype, nullptr, 0, stream, false);
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
  return nvfp4::linear_branch(X, M, W, Y, out_dtype, scratch, NVFP4_NOALLOC_SCRATCH_BYTES, stream, true);
}
