"""nvfp4_linear_noalloc, the linear layer for callers that cannot allocate
device memory (plugins in a host framework that owns every allocation,
runtimes without a device allocator).  It keeps its scratch in an array built
into the library; on consecutive calls that share that array its output must
equal nvfp4_linear's -- the same kernels on the same inputs, so equal bit for
bit, which is within any tolerance the GEMM tests use.

This file is collected last on purpose: if it fails, every other test has
already run.  It passes alone in a fresh process and after the others."""
import ctypes

import pytest

import synth
from nvfp4_testutil import to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import nvfp4_weight_quantized_gb300 as nv  # noqa: E402


@pytest.fixture(scope="module")
def L():
    from nvfp4_weight_quantized_gb300 import build
    build.build()
    return nv.lib()


def _noalloc_raw(L, X, W, out_dtype):
    """Through the C ABI with raw pointers; the caller provides only X, W and Y."""
    M = X.shape[0]
    Y = torch.empty((M, W.N), dtype=torch.float32 if out_dtype == nv.OUT_F32 else torch.bfloat16,
                    device=X.device)
    d = W.descriptor()
    st = L.nvfp4_linear_noalloc(X.data_ptr(), M, ctypes.byref(d), Y.data_ptr(), out_dtype,
                                torch.cuda.current_stream().cuda_stream)
    assert st == nv.OK, L.nvfp4_last_error()
    return Y


def test_noalloc_matches_linear_on_consecutive_calls(L):
    N, K = 1024, 2048
    W = nv.nvfp4_quantize_fos(to_dev(synth.weight_normal(N, K, seed=61, outlier_frac=0.01)))
    old = nv.nvfp4_get_crossover(N, K)
    nv.nvfp4_set_crossover(N, K, 48)
    try:
        # two W4A4 calls in a row (the second reuses the scratch the first left
        # behind), then a W4A16 call, each against nvfp4_linear
        for M, seed, od in ((300, 1, nv.OUT_F32), (130, 2, nv.OUT_BF16), (16, 3, nv.OUT_F32)):
            X = to_dev(synth.act_student_t(M, K, seed=seed))
            y = _noalloc_raw(L, X, W, od)
            ref = nv.nvfp4_linear(X, W, od)
            torch.cuda.synchronize()
            assert torch.equal(y, ref), f"noalloc M={M}: differs from nvfp4_linear"
        assert nv.nvfp4_get_device_status() == nv.OK
    finally:
        nv.nvfp4_set_crossover(N, K, old)


def test_noalloc_rejects_scratch_beyond_its_size(L):
    N, K = 256, 4096
    W = nv.nvfp4_quantize_fos(to_dev(synth.weight_normal(N, K, seed=62)))
    M = 16384  # needs about 38 MB of scratch at K = 4096, above the 32 MiB built in
    assert nv.nvfp4_workspace_bytes(nv.OP_LINEAR, M, N, K) > nv.NOALLOC_SCRATCH_BYTES
    d = W.descriptor()
    st = L.nvfp4_linear_noalloc(None, M, ctypes.byref(d), None, nv.OUT_BF16, None)
    assert st == nv.ERR_WORKSPACE
    msg = L.nvfp4_last_error().decode()
    assert "scratch" in msg and str(M) in msg
