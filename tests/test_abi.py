"""The C ABI without a GPU: the library builds, loads and exports every
function include/nvfp4.h declares; host-only calls and argument checks work
and return their status before anything touches the device."""
import ctypes

import pytest

import nvfp4_weight_quantized_gb300 as nv
from nvfp4_weight_quantized_gb300 import build as nvbuild


@pytest.fixture(scope="module")
def L():
    nvbuild.build()
    return nv.lib()


def test_exports_every_declared_symbol(L):
    names = nv.declared_functions()
    assert {"nvfp4_quantize_fos", "nvfp4_quantize_act", "nvfp4_gemm_w4a16", "nvfp4_gemm_w4a4",
            "nvfp4_linear", "nvfp4_scales_mma_bytes", "nvfp4_workspace_bytes", "nvfp4_set_crossover",
            "nvfp4_get_crossover", "nvfp4_get_device_status", "nvfp4_status_string",
            "nvfp4_last_error"} <= set(names)
    for n in names:
        assert hasattr(L, n), f"{n} declared in nvfp4.h but not exported"


def test_scales_mma_bytes(L):
    assert nv.nvfp4_scales_mma_bytes(128, 64) == 512
    assert nv.nvfp4_scales_mma_bytes(129, 64) == 1024
    assert nv.nvfp4_scales_mma_bytes(4096, 4096) == 32 * 64 * 512 == 4096 * 4096 // 16
    assert nv.nvfp4_scales_mma_bytes(1, 80) == 2 * 512
    assert nv.nvfp4_scales_mma_bytes(0, 64) == 0 and nv.nvfp4_scales_mma_bytes(4, 24) == 0


def test_workspace_bytes(L):
    assert nv.nvfp4_workspace_bytes(nv.OP_QUANTIZE_FOS, 0, 4096, 4096) >= 4096
    assert nv.nvfp4_workspace_bytes(nv.OP_GEMM_W4A16, 8, 4096, 4096) == 0
    lin = nv.nvfp4_workspace_bytes(nv.OP_LINEAR, 1024, 11008, 4096)
    assert lin >= 1024 * 2048 + nv.nvfp4_scales_mma_bytes(1024, 4096)
    assert nv.nvfp4_workspace_bytes(99, 1, 1, 64) == 0
    # gated MLP: the linear workspace plus fp32 [min(M, 1024), N] staging
    lin300 = nv.nvfp4_workspace_bytes(nv.OP_LINEAR, 300, 2 * 11008, 4096)
    assert nv.nvfp4_workspace_bytes(nv.OP_LINEAR_SILU_MUL, 300, 2 * 11008, 4096) == lin300 + 300 * 2 * 11008 * 4
    big = nv.nvfp4_workspace_bytes(nv.OP_LINEAR_SILU_MUL, 5000, 2 * 11008, 4096)
    assert big == nv.nvfp4_workspace_bytes(nv.OP_LINEAR, 5000, 2 * 11008, 4096) + 1024 * 2 * 11008 * 4
    # QAT backward: bf16 W_hat^T [K, Np], X_hat^T [K, Mp], dY^T [N, Mp] (rows padded to 16),
    # each 256-byte aligned, plus a padded dY [M, Np] when N % 8 != 0
    assert nv.nvfp4_workspace_bytes(nv.OP_QAT_BACKWARD, 37, 200, 320) == 320 * 208 * 2 + 320 * 48 * 2 + 200 * 48 * 2
    a256 = lambda v: (v + 255) // 256 * 256  # noqa: E731
    assert nv.nvfp4_workspace_bytes(nv.OP_QAT_BACKWARD, 37, 201, 320) == \
        320 * 208 * 2 + 320 * 48 * 2 + a256(201 * 48 * 2) + a256(37 * 208 * 2)


def test_crossover_table(L):
    default = nv.nvfp4_get_crossover()
    assert default >= 1
    saved = nv.nvfp4_get_crossover(4096, 4096)
    nv.nvfp4_set_crossover(4096, 4096, 17)
    assert nv.nvfp4_get_crossover(4096, 4096) == 17
    assert nv.nvfp4_get_crossover(12345, 4096) == default
    with pytest.raises(nv.NVFP4Error):
        nv.nvfp4_set_crossover(1, 1, -1)
    nv.nvfp4_set_crossover(4096, 4096, saved)


def test_w4a16_kernel_knob(L):
    saved = nv.nvfp4_get_w4a16_rf_max_m()
    assert 0 <= saved <= 64
    nv.nvfp4_set_w4a16_rf_max_m(0)
    assert nv.nvfp4_get_w4a16_rf_max_m() == 0
    for bad in (-1, 65):
        with pytest.raises(nv.NVFP4Error):
            nv.nvfp4_set_w4a16_rf_max_m(bad)
    nv.nvfp4_set_w4a16_rf_max_m(saved)
    assert nv.nvfp4_get_w4a16_rf_max_m() == saved


def test_w4a16_sk_knob(L):
    saved = nv.nvfp4_get_w4a16_sk_max_m()
    assert -1 <= saved <= 64
    for v in (0, 64, -1):
        nv.nvfp4_set_w4a16_sk_max_m(v)
        assert nv.nvfp4_get_w4a16_sk_max_m() == v
    for bad in (-2, 65):
        with pytest.raises(nv.NVFP4Error):
            nv.nvfp4_set_w4a16_sk_max_m(bad)
    nv.nvfp4_set_w4a16_sk_max_m(saved)
    assert nv.nvfp4_get_w4a16_sk_max_m() == saved


def test_w4a4_cluster_knob(L):
    saved = nv.nvfp4_get_w4a4_cluster()
    assert saved in (1, 2)
    for v in (1, 2):
        nv.nvfp4_set_w4a4_cluster(v)
        assert nv.nvfp4_get_w4a4_cluster() == v
    for bad in (0, 3, 4, 8):
        with pytest.raises(nv.NVFP4Error):
            nv.nvfp4_set_w4a4_cluster(bad)
    nv.nvfp4_set_w4a4_cluster(saved)


def test_act_fos_knob(L):
    saved = nv.nvfp4_get_act_fos()
    for v in (True, False):
        nv.nvfp4_set_act_fos(v)
        assert nv.nvfp4_get_act_fos() == v
    nv.nvfp4_set_act_fos(saved)


def test_status_strings(L):
    for s in range(9):
        assert nv.nvfp4_status_string(s)
    assert "unknown" in nv.nvfp4_status_string(123)


FAKE = 0x100000  # a 16-byte aligned host-side integer; never dereferenced


def _q(L, W=FAKE, N=4, K=64, codes=FAKE, scales=FAKE, smma=FAKE, ts=FAKE, choice=None, m4=None,
       ws=FAKE, wsb=1 << 20):
    return L.nvfp4_quantize_fos(W, N, K, 0.0, codes, scales, smma, ts, choice, m4, ws, wsb, None)


def test_quantize_argument_errors(L):
    assert _q(L, W=None) == nv.ERR_INVALID_ARG
    assert _q(L, codes=None) == nv.ERR_INVALID_ARG
    assert _q(L, ts=None) == nv.ERR_INVALID_ARG
    assert _q(L, scales=None, smma=None) == nv.ERR_INVALID_ARG
    assert _q(L, K=24) == nv.ERR_SHAPE
    assert _q(L, K=0) == nv.ERR_SHAPE
    assert _q(L, N=0) == nv.ERR_SHAPE
    assert _q(L, N=-3) == nv.ERR_SHAPE
    assert _q(L, W=FAKE + 8) == nv.ERR_ALIGN
    assert _q(L, codes=FAKE + 4) == nv.ERR_ALIGN
    assert _q(L, ts=FAKE + 2) == nv.ERR_ALIGN
    assert _q(L, ws=None) == nv.ERR_WORKSPACE
    assert _q(L, wsb=16) == nv.ERR_WORKSPACE
    assert L.nvfp4_quantize_act(FAKE, 2, 40, 0.0, FAKE, None, FAKE, FAKE, FAKE, 1 << 20, None) == nv.ERR_SHAPE
    assert L.nvfp4_last_error()


def _w(codes=FAKE, smma=FAKE, ts=FAKE, N=256, K=512):
    return nv._Weight(codes, smma, ts, N, K)


def test_gemm_argument_errors(L):
    g16 = L.nvfp4_gemm_w4a16
    assert g16(FAKE, 4, None, FAKE, 0, None, 0, None) == nv.ERR_INVALID_ARG
    assert g16(FAKE, 4, ctypes.byref(_w(codes=None)), FAKE, 0, None, 0, None) == nv.ERR_INVALID_ARG
    assert g16(FAKE, 4, ctypes.byref(_w(K=40)), FAKE, 0, None, 0, None) == nv.ERR_SHAPE  # K % 16
    assert g16(FAKE, 4, ctypes.byref(_w(N=0)), FAKE, 0, None, 0, None) == nv.ERR_SHAPE
    assert g16(FAKE, 4, ctypes.byref(_w(codes=FAKE + 1)), FAKE, 0, None, 0, None) == nv.ERR_ALIGN
    assert g16(FAKE, -1, ctypes.byref(_w()), FAKE, 0, None, 0, None) == nv.ERR_SHAPE
    assert g16(FAKE, 4, ctypes.byref(_w()), FAKE, 7, None, 0, None) == nv.ERR_INVALID_ARG
    assert g16(FAKE + 8, 4, ctypes.byref(_w()), FAKE, 0, None, 0, None) == nv.ERR_ALIGN
    assert g16(None, 4, ctypes.byref(_w()), FAKE, 0, None, 0, None) == nv.ERR_INVALID_ARG
    # M == 0 is a no-op that succeeds without touching the device
    assert g16(None, 0, ctypes.byref(_w()), None, 0, None, 0, None) == nv.OK
    g4 = L.nvfp4_gemm_w4a4
    assert g4(None, FAKE, FAKE, 4, ctypes.byref(_w()), FAKE, 0, None, 0, None) == nv.ERR_INVALID_ARG
    assert g4(FAKE, FAKE, FAKE + 2, 4, ctypes.byref(_w()), FAKE, 0, None, 0, None) == nv.ERR_ALIGN
    assert g4(FAKE, FAKE, FAKE, 0, ctypes.byref(_w()), None, 0, None, 0, None) == nv.OK
    # the FP4 MMA's K step: W4A16 takes K = 48, W4A4 does not
    assert g4(FAKE, FAKE, FAKE, 4, ctypes.byref(_w(K=48)), FAKE, 0, None, 0, None) == nv.ERR_SHAPE


def test_linear_workspace_errors(L):
    nv.nvfp4_set_crossover(256, 512, 8)
    try:
        lin = L.nvfp4_linear
        # above the crossover the W4A4 branch needs the workspace
        assert lin(FAKE, 100, ctypes.byref(_w()), FAKE, 0, None, 0, None) == nv.ERR_WORKSPACE
        assert lin(FAKE, 100, ctypes.byref(_w()), FAKE, 0, FAKE + 16, 1 << 30, None) == nv.ERR_WORKSPACE
        assert lin(FAKE, 100, ctypes.byref(_w()), FAKE, 0, FAKE, 16, None) == nv.ERR_WORKSPACE
    finally:
        nv.nvfp4_set_crossover(256, 512, nv.nvfp4_get_crossover())


def test_product_path_has_no_oracle_dependency():
    """The binding and the CUDA sources never load the oracle."""
    import glob
    import os
    import re
    pkg = os.path.dirname(nv.__file__)
    pat = re.compile(r"^\s*(import\s+oracle|from\s+oracle)|liboracle|nvfp4_oracle|oracle/", re.M)
    for path in glob.glob(os.path.join(pkg, "**", "*"), recursive=True):
        if path.endswith((".py", ".cu", ".cuh", ".h")):
            assert not pat.search(open(path).read()), path


def test_new_call_argument_errors(L):
    """Argument checks of the gated-MLP, GPTQ, dequantisation and QAT calls
    return before any device work."""
    sm = L.nvfp4_linear_silu_mul
    assert sm(FAKE, 4, ctypes.byref(_w(N=255)), FAKE, 0, FAKE, 1 << 30, None) == nv.ERR_SHAPE  # odd N
    assert sm(FAKE, -1, ctypes.byref(_w()), FAKE, 0, FAKE, 1 << 30, None) == nv.ERR_SHAPE
    assert sm(None, 4, ctypes.byref(_w()), FAKE, 0, FAKE, 1 << 30, None) == nv.ERR_INVALID_ARG
    assert sm(FAKE + 8, 4, ctypes.byref(_w()), FAKE, 0, FAKE, 1 << 30, None) == nv.ERR_ALIGN
    assert sm(FAKE, 4, ctypes.byref(_w()), FAKE, 0, FAKE, 16, None) == nv.ERR_WORKSPACE
    assert sm(FAKE, 4, ctypes.byref(_w()), FAKE, 9, FAKE, 1 << 30, None) == nv.ERR_INVALID_ARG
    assert sm(None, 0, ctypes.byref(_w()), None, 0, None, 0, None) == nv.OK
    gq = L.nvfp4_gptq_fos
    assert gq(FAKE, 64, 256, None, 0.01, FAKE, None, FAKE, FAKE, FAKE, 1 << 30, None) == nv.ERR_INVALID_ARG
    assert gq(FAKE, 64, 256, FAKE, -1.0, FAKE, None, FAKE, FAKE, FAKE, 1 << 30, None) == nv.ERR_INVALID_ARG
    assert gq(FAKE, 64, 250, FAKE, 0.01, FAKE, None, FAKE, FAKE, FAKE, 1 << 30, None) == nv.ERR_SHAPE
    assert gq(FAKE, 64, 16384, FAKE, 0.01, FAKE, None, FAKE, FAKE, FAKE, 1 << 40, None) == nv.ERR_SHAPE
    assert gq(FAKE, 64, 256, FAKE + 4, 0.01, FAKE, None, FAKE, FAKE, FAKE, 1 << 30, None) == nv.ERR_ALIGN
    assert gq(FAKE, 64, 256, FAKE, 0.01, FAKE, None, FAKE, FAKE, FAKE, 1024, None) == nv.ERR_WORKSPACE
    dq = L.nvfp4_dequantize
    assert dq(None, FAKE, FAKE, 4, 64, FAKE, None) == nv.ERR_INVALID_ARG
    assert dq(FAKE, FAKE, FAKE, 4, 40, FAKE, None) == nv.ERR_SHAPE
    assert dq(FAKE, FAKE, FAKE, 4, 64, FAKE + 2, None) == nv.ERR_ALIGN
    assert dq(FAKE, FAKE, FAKE, 0, 64, FAKE, None) == nv.OK
    qb = L.nvfp4_qat_backward
    assert qb(FAKE, 4, ctypes.byref(_w()), None, None, None, None, None, FAKE, 1 << 30, None) == nv.OK  # nothing asked
    assert qb(None, 4, ctypes.byref(_w()), None, None, None, FAKE, None, FAKE, 1 << 30, None) == nv.ERR_INVALID_ARG
    assert qb(FAKE, 4, ctypes.byref(_w()), None, None, None, None, FAKE, FAKE, 1 << 30, None) == nv.ERR_INVALID_ARG
    assert qb(FAKE, 4, ctypes.byref(_w()), None, None, None, FAKE, None, FAKE, 16, None) == nv.ERR_WORKSPACE


def test_crossover_rule_from_timings():
    """The tuner's rule on hand-made timings {M: (t_w4a16, t_w4a4)}: the
    largest M where W4A16 is no slower, scanning up until W4A4 wins twice
    in a row (one noisy loss does not end the scan)."""
    from nvfp4_weight_quantized_gb300.tune import crossover_from
    assert crossover_from({1: (1, 2), 8: (1, 2), 16: (3, 2), 32: (3, 2), 48: (1, 2)}) == 8
    assert crossover_from({1: (1, 2), 8: (3, 2), 16: (1, 2), 32: (3, 2), 64: (3, 2)}) == 16
    assert crossover_from({1: (2, 2), 4: (2, 2)}) == 4        # a tie keeps W4A16
    assert crossover_from({1: (3, 2), 2: (3, 2), 4: (1, 2)}) == 0
    assert crossover_from({64: (1, 2), 1: (3, 2), 8: (1, 2)}) == 64  # keys are sorted


def test_noalloc_argument_paths(L):
    """nvfp4_linear_noalloc reports argument errors, accepts M == 0 and
    rejects scratch needs beyond its built-in array, all before any device
    call (no GPU here)."""
    na = L.nvfp4_linear_noalloc
    assert na(FAKE, 4, None, FAKE, 0, None) == nv.ERR_INVALID_ARG
    assert na(FAKE, 4, ctypes.byref(_w(K=40)), FAKE, 0, None) == nv.ERR_SHAPE
    assert na(FAKE, -2, ctypes.byref(_w()), FAKE, 0, None) == nv.ERR_SHAPE
    assert na(None, 0, ctypes.byref(_w()), None, 0, None) == nv.OK
    big = _w(N=256, K=4096)
    M = 16384
    assert nv.nvfp4_workspace_bytes(nv.OP_LINEAR, M, 256, 4096) > nv.NOALLOC_SCRATCH_BYTES
    assert na(FAKE, M, ctypes.byref(big), FAKE, 0, None) == nv.ERR_WORKSPACE
    assert b"scratch" in L.nvfp4_last_error()


def test_binding_declares_every_signature(L):
    """Every function of the header has its argument and result types set in
    the binding (an unset signature would pass 64-bit sizes as C ints)."""
    for n in nv.declared_functions():
        assert getattr(L, n).argtypes is not None, f"{n}: no ctypes signature in the binding"


def test_measure_fp4_mma_argument_errors(L):
    """nvfp4_measure_fp4_mma rejects bad arguments before touching a device."""
    import ctypes
    pairs = ctypes.c_int(7)
    fn = L.nvfp4_measure_fp4_mma
    assert fn(0, ctypes.c_void_p(16), 4, ctypes.byref(pairs), None) == nv.ERR_INVALID_ARG
    assert fn(10, None, 4, ctypes.byref(pairs), None) == nv.ERR_INVALID_ARG
    assert fn(10, ctypes.c_void_p(16), 0, ctypes.byref(pairs), None) == nv.ERR_INVALID_ARG
    assert fn(10, ctypes.c_void_p(16), 4, None, None) == nv.ERR_INVALID_ARG


def test_single_launch_quantizer_knob(L):
    saved = nv.nvfp4_get_single_launch_quantizer()
    for v in (False, True):
        nv.nvfp4_set_single_launch_quantizer(v)
        assert nv.nvfp4_get_single_launch_quantizer() == v
    nv.nvfp4_set_single_launch_quantizer(saved)
