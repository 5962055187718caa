"""GPTQ inside FourOverSix scales on the GPU against the oracle: the codes,
scales and tensor scale bit for bit (both sides take the same binary32 steps
in the same order)."""
import numpy as np
import pytest

import oracle
import synth
from nvfp4_testutil import to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import nvfp4_weight_quantized_gb300 as nv  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    from nvfp4_weight_quantized_gb300 import build
    build.build()
    nv.lib()


def _hessian(K, T, seed):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((T, K)).astype(np.float32)
    X[:, : K // 4] *= 3.0
    return (2.0 * X.T @ X / T).astype(np.float32)


@pytest.mark.parametrize("NK", [(256, 512), (200, 384), (64, 1040)])
def test_gptq_fos_bit_exact(NK):
    """Several 128-column blocks, a ragged last block (K = 1040) and rows that
    do not fill the last 128-row CTA (N = 200)."""
    N, K = NK
    w = synth.weight_normal(N, K, seed=N + K, outlier_frac=0.01)
    H = _hessian(K, 2 * K, seed=K)
    q = nv.nvfp4_gptq_fos(to_dev(w), torch.from_numpy(H).cuda())
    torch.cuda.synchronize()
    assert nv.nvfp4_get_device_status() == 0
    ref = oracle.gptq_fos(w, H, damp=0.01, block=128)
    assert float(q.tensor_scale.item()) == ref["ts"]
    assert np.array_equal(q.scales.cpu().numpy(), ref["scales"])
    assert np.array_equal(q.scales_mma.cpu().numpy(), oracle.scales_to_mma(ref["scales"], K))
    got = q.codes.cpu().numpy()
    assert np.array_equal(got, ref["codes"]), f"{int((got != ref['codes']).sum())} code bytes differ"


def test_gptq_identity_hessian_is_fos_rtn():
    N, K = 128, 256
    w = synth.weight_normal(N, K, seed=31, outlier_frac=0.02)
    q = nv.nvfp4_gptq_fos(to_dev(w), torch.eye(K, device="cuda"))
    f = nv.nvfp4_quantize_fos(to_dev(w))
    torch.cuda.synchronize()
    assert torch.equal(q.codes, f.codes) and torch.equal(q.scales_mma, f.scales_mma)


def test_gptq_not_positive_definite_sets_status():
    N, K = 32, 64
    w = synth.weight_normal(N, K, seed=32)
    nv.nvfp4_gptq_fos(to_dev(w), -torch.eye(K, device="cuda"))
    torch.cuda.synchronize()
    st = nv.nvfp4_get_device_status()
    assert st != 0
    assert nv.nvfp4_get_device_status() == 0  # read and cleared
