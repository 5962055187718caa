"""nvfp4_linear: the M-based dispatch between the W4A16 and W4A4 paths, end
to end from bf16 activations, against the oracle and against the two paths
called directly."""
import numpy as np
import pytest

import oracle
import synth
from nvfp4_testutil import (THREADS, assert_gemm_close, assert_silu_mul_close, oracle_w4a16, oracle_w4a4,
                            to_dev, y_to_np)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import nvfp4_weight_quantized_gb300 as nv  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    from nvfp4_weight_quantized_gb300 import build
    build.build()
    nv.lib()


def test_dispatch_follows_crossover():
    N, K = 384, 1024
    w = synth.weight_normal(N, K, seed=91, outlier_frac=0.01)
    W = nv.nvfp4_quantize_fos(to_dev(w))
    old = nv.nvfp4_get_crossover(N, K)
    nv.nvfp4_set_crossover(N, K, 40)
    try:
        for M in (1, 40, 41, 200):
            x = synth.act_student_t(M, K, seed=M)
            X = to_dev(x)
            y = nv.nvfp4_linear(X, W, nv.OUT_F32)
            if M <= 40:
                direct = nv.nvfp4_gemm_w4a16(X, W, nv.OUT_F32)
            else:
                direct = nv.nvfp4_gemm_w4a4(nv.nvfp4_quantize_act(X), W, nv.OUT_F32)
            torch.cuda.synchronize()
            assert torch.equal(y, direct), M
            # end to end against the oracle on the same path
            wts = oracle.tensor_scale(w)
            wref = oracle.quantize_rows(w, wts, True, THREADS)
            if M <= 40:
                ref = oracle_w4a16(x, wref["codes"], wref["scales"], wref["ts"])
            else:
                aref = oracle.quantize_rows(x, oracle.tensor_scale(x), False, THREADS)
                ref = oracle_w4a4(aref["codes"], aref["scales"], aref["ts"], wref["codes"], wref["scales"],
                                  wref["ts"])
            assert_gemm_close(y_to_np(y), ref, bf16=False, what=f"linear M={M}")
    finally:
        nv.nvfp4_set_crossover(N, K, old)


def test_linear_with_fos_activations():
    """With the activation FourOverSix option the W4A4 branch equals W4A4 on
    nvfp4_quantize_fos(X) and matches the oracle with FourOverSix-quantised
    activations; the W4A16 branch is unaffected."""
    N, K = 384, 1024
    w = synth.weight_normal(N, K, seed=93, outlier_frac=0.01)
    W = nv.nvfp4_quantize_fos(to_dev(w))
    wts = oracle.tensor_scale(w)
    wref = oracle.quantize_rows(w, wts, True, THREADS)
    old = nv.nvfp4_get_crossover(N, K)
    nv.nvfp4_set_crossover(N, K, 40)
    nv.nvfp4_set_act_fos(True)
    try:
        for M in (1, 41, 130, 300):
            x = synth.act_student_t(M, K, seed=700 + M)
            X = to_dev(x)
            y = nv.nvfp4_linear(X, W, nv.OUT_F32)
            if M <= 40:
                direct = nv.nvfp4_gemm_w4a16(X, W, nv.OUT_F32)
            else:
                q = nv.nvfp4_quantize_fos(X, logical_scales=False, choice=False)
                A = nv.NVFP4Act(codes=q.codes, scales_mma=q.scales_mma, tensor_scale=q.tensor_scale, M=M, K=K)
                direct = nv.nvfp4_gemm_w4a4(A, W, nv.OUT_F32)
            torch.cuda.synchronize()
            assert torch.equal(y, direct), M
            if M > 40:
                aref = oracle.quantize_rows(x, oracle.tensor_scale(x), True, THREADS)
                ref = oracle_w4a4(aref["codes"], aref["scales"], aref["ts"], wref["codes"], wref["scales"],
                                  wref["ts"])
                assert_gemm_close(y_to_np(y), ref, bf16=False, what=f"linear act-FOS M={M}")
    finally:
        nv.nvfp4_set_act_fos(False)
        nv.nvfp4_set_crossover(N, K, old)


def test_linear_small_k_always_takes_w4a16():
    N, K = 64, 128  # below one 256-wide K stage of the tensor-core kernel
    w = synth.weight_normal(N, K, seed=5)
    W = nv.nvfp4_quantize_fos(to_dev(w))
    x = to_dev(synth.act_normal(300, K, seed=6))
    y = nv.nvfp4_linear(x, W, nv.OUT_F32)
    assert torch.equal(y, nv.nvfp4_gemm_w4a16(x, W, nv.OUT_F32))


def test_default_crossover_is_sane():
    c = nv.nvfp4_get_crossover()
    assert 1 <= c <= 4096


def _gate_up_refs(x, wref, path_w4a4, m_rows=None):
    """binary64 G and U for a gate/up weight [2F, K] on the given path."""
    if path_w4a4:
        aref = oracle.quantize_rows(x, oracle.tensor_scale(x), False, THREADS)
        y = oracle_w4a4(aref["codes"], aref["scales"], aref["ts"], wref["codes"], wref["scales"], wref["ts"],
                        m_rows=m_rows)
    else:
        y = oracle_w4a16(x if m_rows is None else x[m_rows], wref["codes"], wref["scales"], wref["ts"])
    F = y.y.shape[1] // 2
    return y.cols(slice(0, F)), y.cols(slice(F, None))


@pytest.mark.parametrize("F", [256, 384, 200])
def test_linear_silu_mul(F):
    """Gated MLP projection against the oracle on both paths: W4A16 (M <= 40)
    with the separate silu kernel; W4A4 with silu(G) * U fused into the GEMM's
    epilogue for bf16 output and F % 128 == 0 (CTA pairs above 128 tokens,
    single CTAs up to 128 or when pairs are off), separate otherwise (fp32
    output, F = 200)."""
    K = 1024
    N = 2 * F
    w = synth.weight_normal(N, K, seed=F + 17, outlier_frac=0.01)
    W = nv.nvfp4_quantize_fos(to_dev(w))
    wref = oracle.quantize_rows(w, oracle.tensor_scale(w), True, THREADS)
    old = nv.nvfp4_get_crossover(N, K)
    saved_cl = nv.nvfp4_get_w4a4_cluster()
    nv.nvfp4_set_crossover(N, K, 40)
    try:
        for M in (1, 40, 41, 128, 130, 300):
            x = synth.act_student_t(M, K, seed=900 + M)
            X = to_dev(x)
            g, u = _gate_up_refs(x, wref, M > 40)
            for od in (nv.OUT_BF16, nv.OUT_F32):
                for ctas in ((2, 1) if M > 128 else (2,)):
                    nv.nvfp4_set_w4a4_cluster(ctas)
                    y = y_to_np(nv.nvfp4_linear_silu_mul(X, W, od))
                    torch.cuda.synchronize()
                    assert_silu_mul_close(y, g, u, bf16=od == nv.OUT_BF16, what=f"F={F} M={M} od={od} ctas={ctas}")
        assert nv.nvfp4_get_device_status() == 0
    finally:
        nv.nvfp4_set_w4a4_cluster(saved_cl)
        nv.nvfp4_set_crossover(N, K, old)


def test_linear_silu_mul_chunks_and_fused_match():
    """More rows than one 1024-row workspace chunk on the separate path (fp32
    output), sampled against the oracle; the fused bf16 result equals the
    separate path's bf16 rounding of the same binary32 expression within one
    bf16 step."""
    F, K, M = 256, 512, 1100
    N = 2 * F
    w = synth.weight_normal(N, K, seed=4242, outlier_frac=0.01)
    W = nv.nvfp4_quantize_fos(to_dev(w))
    wref = oracle.quantize_rows(w, oracle.tensor_scale(w), True, THREADS)
    x = synth.act_student_t(M, K, seed=4243)
    X = to_dev(x)
    rows = np.array(sorted(set(range(0, M, 37)) | {0, 1023, 1024, M - 1}))
    g, u = _gate_up_refs(x, wref, True, m_rows=rows)
    y32 = y_to_np(nv.nvfp4_linear_silu_mul(X, W, nv.OUT_F32))
    assert_silu_mul_close(y32[rows], g, u, bf16=False, what="chunked fp32")
    fused = nv.nvfp4_linear_silu_mul(X, W, nv.OUT_BF16).float()
    sep = torch.from_numpy(y32).cuda().to(torch.bfloat16).float()
    torch.cuda.synchronize()
    diff = (fused - sep).abs()
    step = sep.abs() * 2.0 ** -7 + 2.0 ** -133
    assert bool((diff <= step).all()), float((diff / step).max())
