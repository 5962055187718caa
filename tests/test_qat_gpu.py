"""NVFP4 dequantisation and the straight-through backward pass of the
FP4-forward linear layer (quantisation-aware training) on the GPU, against
the oracle."""
import numpy as np
import pytest

import oracle
import synth
from nvfp4_testutil import THREADS, assert_gemm_close, oracle_qat, to_dev, y_to_np

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import nvfp4_weight_quantized_gb300 as nv  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    from nvfp4_weight_quantized_gb300 import build
    build.build()
    nv.lib()


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("shape", [(1, 16), (130, 320), (256, 4096), (300, 1024)])
def test_dequantize_bit_exact(shape):
    R, K = shape
    w = synth.weight_normal(R, K, seed=R + K, outlier_frac=0.02)
    q = nv.nvfp4_quantize_fos(to_dev(w))
    got = _bits(nv.nvfp4_dequantize(q.codes, q.scales_mma, q.tensor_scale, R, K))
    ref = oracle.quantize_fos(w)
    want = oracle.dequant_bf16(ref["codes"], ref["scales"], ref["ts"])
    assert np.array_equal(got, want)


@pytest.mark.parametrize("MNK", [(1, 64, 64), (37, 200, 320), (20, 100, 192), (300, 512, 1024), (260, 520, 576)])
def test_qat_backward(MNK):
    """dX = dY W_hat (bf16) and dW = dY^T X_hat (fp32) against the binary64
    oracle on the same bf16 operands (GEMM tolerance: fp32 accumulation).
    The shapes cover rows padded to 16 (M = 1, 37, 20, 260), dY rows that are
    not 16-byte aligned (N = 100: a padded copy), more than one 256 x 256
    output tile each way and a ragged last one."""
    M, N, K = MNK
    w = synth.weight_normal(N, K, seed=N + 3 * K, outlier_frac=0.01)
    x = synth.act_student_t(M, K, seed=M + 5)
    rng = np.random.default_rng(M * 7 + N)
    dy = synth.f32_to_bf16_bits(rng.standard_normal((M, N)).astype(np.float32))
    W = nv.nvfp4_quantize_fos(to_dev(w))
    A = nv.nvfp4_quantize_act(to_dev(x))
    dX, dW = nv.nvfp4_qat_backward(to_dev(dy), W, A)
    torch.cuda.synchronize()
    wref = oracle.quantize_fos(w)
    aref = oracle.quantize_rows(x, oracle.tensor_scale(x), False, THREADS)
    w_hat = oracle.dequant_bf16(wref["codes"], wref["scales"], wref["ts"])
    x_hat = oracle.dequant_bf16(aref["codes"], aref["scales"], aref["ts"])
    dx_ref, dw_ref = oracle_qat(dy, w_hat, x_hat)
    assert_gemm_close(y_to_np(dX), dx_ref, bf16=True, what=f"dX {MNK}")
    assert_gemm_close(dW.cpu().numpy().astype(np.float64), dw_ref, bf16=False, what=f"dW {MNK}")
    # either gradient alone
    dX2, none = nv.nvfp4_qat_backward(to_dev(dy), W, None, want_dw=False)
    assert none is None and torch.equal(dX2, dX)
    none, dW2 = nv.nvfp4_qat_backward(to_dev(dy), W, A, want_dx=False)
    assert none is None and torch.equal(dW2, dW)


def test_dequantize_ties_by_hand():
    """The oracle's by-hand round-to-nearest-even cases on the GPU: block
    scale 0x38 (value 1), codes +-1 or +-1.5, tensor scales that make the
    binary32 product a bf16 midpoint (exactly, or after a binary32 tie)."""
    cases = [(0x02 | (0x0A << 4), 1.0 + 2.0 ** -8, 0x3F80),
             (0x02 | (0x0A << 4), 1.0 + 3 * 2.0 ** -8, 0x3F82),
             (0x03 | (0x0B << 4), 11228502 * 2.0 ** -24, 0x3F80)]
    smma = np.zeros(512, np.uint8)  # one 128 x 4 scale tile; scale (0, 0) at byte 0
    smma[0] = 0x38
    for byte, ts, want in cases:
        codes = np.array([[byte] + [0] * 7], np.uint8)
        Y = nv.nvfp4_dequantize(torch.from_numpy(codes).cuda(), torch.from_numpy(smma).cuda(),
                                torch.tensor([ts], dtype=torch.float32, device="cuda"), 1, 16)
        got = _bits(Y)[0]
        assert list(got[:2]) == [want, want | 0x8000] and not got[2:].any(), (hex(byte), ts)
        assert np.array_equal(got, oracle.dequant_bf16(codes, np.array([[0x38]], np.uint8), ts)[0])
