"""W4A16 and W4A4 GEMMs on the GPU against the binary64 oracle.

The GEMMs are fed operands quantised by the oracle, so these tests check the
GEMM kernels alone (the quantisers have their own bit-exact tests)."""
import numpy as np
import pytest

import oracle
import synth
from nvfp4_testutil import THREADS, assert_gemm_close, oracle_w4a16, oracle_w4a4, to_dev, y_to_np

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import nvfp4_weight_quantized_gb300 as nv  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    from nvfp4_weight_quantized_gb300 import build
    build.build()
    nv.lib()


def oracle_weight(w_bits):
    ts = oracle.tensor_scale(w_bits)
    return oracle.quantize_rows(w_bits, ts, True, THREADS)


def oracle_act(x_bits):
    ts = oracle.tensor_scale(x_bits)
    return oracle.quantize_rows(x_bits, ts, False, THREADS)


def dev_weight(ref, K):
    N = ref["codes"].shape[0]
    return nv.NVFP4Weight(
        codes=torch.from_numpy(ref["codes"]).cuda(),
        scales_mma=torch.from_numpy(oracle.scales_to_mma(ref["scales"], K)).cuda(),
        tensor_scale=torch.tensor([ref["ts"]], dtype=torch.float32).cuda(), N=N, K=K)


def dev_act(ref, K):
    M = ref["codes"].shape[0]
    return nv.NVFP4Act(
        codes=torch.from_numpy(ref["codes"]).cuda(),
        scales_mma=torch.from_numpy(oracle.scales_to_mma(ref["scales"], K)).cuda(),
        tensor_scale=torch.tensor([ref["ts"]], dtype=torch.float32).cuda(), M=M, K=K)


def sample_rows(n, k, seed):
    rng = np.random.default_rng(seed)
    if k >= n:
        return np.arange(n)
    s = set(rng.choice(n, size=k - 4, replace=False).tolist()) | {0, 1, n - 2, n - 1}
    return np.array(sorted(s))


def run_w4a16(x_bits, wref, K, out_dtype=nv.OUT_BF16, n_rows=None):
    W = dev_weight(wref, K)
    y = nv.nvfp4_gemm_w4a16(to_dev(x_bits), W, out_dtype)
    torch.cuda.synchronize()
    y = y_to_np(y)
    ref = oracle_w4a16(x_bits, wref["codes"], wref["scales"], wref["ts"], n_rows=n_rows)
    if n_rows is not None:
        y = y[:, n_rows]
    return assert_gemm_close(y, ref, bf16=out_dtype == nv.OUT_BF16, what=f"w4a16 M={x_bits.shape[0]}")


def run_w4a4(x_bits, wref, K, out_dtype=nv.OUT_BF16, m_rows=None, n_rows=None):
    aref = oracle_act(x_bits)
    W = dev_weight(wref, K)
    A = dev_act(aref, K)
    y = y_to_np(nv.nvfp4_gemm_w4a4(A, W, out_dtype))
    torch.cuda.synchronize()
    ref = oracle_w4a4(aref["codes"], aref["scales"], aref["ts"], wref["codes"], wref["scales"], wref["ts"],
                      m_rows=m_rows, n_rows=n_rows)
    if m_rows is not None:
        y = y[m_rows]
    if n_rows is not None:
        y = y[:, n_rows]
    return assert_gemm_close(y, ref, bf16=out_dtype == nv.OUT_BF16, what=f"w4a4 M={x_bits.shape[0]}")


# ----------------------------------------------------------------- W4A16 ---

def test_w4a16_tiny_case():
    w, x = synth.tiny_case()
    wref = oracle_weight(w)
    for od in (nv.OUT_BF16, nv.OUT_F32):
        run_w4a16(x, wref, 512, od)


@pytest.mark.parametrize("shape", [(200, 320), (1, 64), (129, 1024), (256, 4160)])
@pytest.mark.parametrize("M", [1, 5, 13, 64, 70, 129])
def test_w4a16_ragged(shape, M):
    N, K = shape
    wref = oracle_weight(synth.weight_normal(N, K, seed=N + K, outlier_frac=0.01))
    x = synth.act_normal(M, K, seed=M)
    run_w4a16(x, wref, K, nv.OUT_F32)
    run_w4a16(x, wref, K, nv.OUT_BF16)


def each_w4a16_kernel(fn):
    """Runs fn() with each W4A16 kernel forced in turn: the persistent
    split-K kernel, the cluster split kernel and the tensor-memory kernel."""
    saved = (nv.nvfp4_get_w4a16_sk_max_m(), nv.nvfp4_get_w4a16_rf_max_m())
    try:
        for sk, rf in ((64, 64), (0, 64), (0, 0)):
            nv.nvfp4_set_w4a16_sk_max_m(sk)
            nv.nvfp4_set_w4a16_rf_max_m(rf)
            fn()
    finally:
        nv.nvfp4_set_w4a16_sk_max_m(saved[0])
        nv.nvfp4_set_w4a16_rf_max_m(saved[1])


@pytest.mark.parametrize("M", [1, 8, 9, 17, 24, 31, 40, 48, 56, 64])
def test_w4a16_both_kernels(M):
    """Every W4A16 kernel (the decode ones at every token-tile width they are
    built for), forced in turn, matches the oracle."""
    N, K = 328, 1344
    wref = oracle_weight(synth.weight_normal(N, K, seed=77, outlier_frac=0.01))
    x = synth.act_normal(M, K, seed=500 + M)

    def check():
        run_w4a16(x, wref, K, nv.OUT_F32)
        run_w4a16(x, wref, K, nv.OUT_BF16)
    each_w4a16_kernel(check)


@pytest.mark.parametrize("shape", [(128, 256), (128, 64), (256, 4096), (1280, 2048), (200, 11008), (3000, 320)])
@pytest.mark.parametrize("M", [1, 3, 16, 33])
def test_w4a16_split_shapes(shape, M):
    """K splits of every kind: one tile with one stage, one tile split over a
    whole cluster, uneven splits, a ragged last stage, a ragged last tile,
    many tiles."""
    N, K = shape
    wref = oracle_weight(synth.weight_normal(N, K, seed=N + 3 * K, outlier_frac=0.01))
    x = synth.act_normal(M, K, seed=40 + M)
    each_w4a16_kernel(lambda: run_w4a16(x, wref, K, nv.OUT_F32))
    assert nv.nvfp4_get_device_status() == 0


@pytest.mark.parametrize("M", [8, 20])
def test_w4a16_activation_range(M):
    """Tokens spanning the whole bf16 range (tiny, subnormal, huge, zero, a
    token whose magnitude jumps by 2^23 in a later K stage, one that shrinks)
    match the oracle row by row: no kernel loses them to overflow, underflow
    or a per-token power-of-two scaling of the activations."""
    N, K = 328, 1344
    wref = oracle_weight(synth.weight_normal(N, K, seed=78, outlier_frac=0.01))
    rng = np.random.default_rng(600 + M)
    x = rng.standard_normal((M, K))
    x[0] *= 2.0 ** -120                       # tiny (bf16 normal range)
    x[1] *= 2.0 ** 100                        # huge
    x[2, :700] *= 1e-3                        # grows by ~2^23 after the first stages
    x[2, 700:] *= 1e4
    x[3] = 0.0                                # zero token
    x[4, :300] *= 1e6                         # shrinks: later elements far below the maximum
    x[4, 300:] *= 1e-2
    x[5] *= 2.0 ** -130                       # bf16 subnormals only
    x[6, 1000] = 1e36                         # one huge element in an ordinary token
    bits = synth.f32_to_bf16_bits(x.astype(np.float32))

    def check():
        run_w4a16(bits, wref, K, nv.OUT_F32)
        run_w4a16(bits, wref, K, nv.OUT_BF16)
    each_w4a16_kernel(check)


def test_w4a16_weight_prefetch_chain():
    """Back-to-back GEMMs with weight prefetch on (each kernel starts reading
    its weights while the previous one runs) give the same results."""
    shapes = [(384, 1024), (200, 2048), (640, 1024)]
    wrefs = [oracle_weight(synth.weight_normal(N, K, seed=900 + i, outlier_frac=0.01))
             for i, (N, K) in enumerate(shapes)]
    Ws = [dev_weight(w, K) for w, (N, K) in zip(wrefs, shapes)]
    torch.cuda.synchronize()
    saved = nv.nvfp4_get_weight_prefetch()
    try:
        nv.nvfp4_set_weight_prefetch(True)
        for M in (1, 16, 40):
            xs = [synth.act_normal(M, K, seed=950 + M + i) for i, (N, K) in enumerate(shapes)]
            ys = [nv.nvfp4_gemm_w4a16(to_dev(x), W, nv.OUT_F32) for x, W in zip(xs, Ws)]
            torch.cuda.synchronize()
            for x, y, w in zip(xs, ys, wrefs):
                ref = oracle_w4a16(x, w["codes"], w["scales"], w["ts"])
                assert_gemm_close(y_to_np(y), ref, bf16=False, what=f"prefetch M={M}")
    finally:
        nv.nvfp4_set_weight_prefetch(saved)
    assert nv.nvfp4_get_device_status() == 0


def test_w4a16_decode_shapes():
    wref = oracle_weight(synth.decode_weight())
    cols = sample_rows(4096, 384, 1)
    for M in synth.DECODE_M:
        worst = run_w4a16(synth.decode_act(M), wref, 4096, nv.OUT_BF16, n_rows=cols)
        worst32 = run_w4a16(synth.decode_act(M), wref, 4096, nv.OUT_F32, n_rows=cols)
        print(f"decode M={M}: worst normwise rel err bf16 {worst:.2e} fp32 {worst32:.2e}")


def test_w4a16_mlp_shapes():
    gate_up, down = synth.mlp_weights()
    for w, K, seed in ((gate_up, 4096, 310), (down, 11008, 311)):
        wref = oracle_weight(w)
        cols = sample_rows(w.shape[0], 256, seed)
        for M in synth.MLP_M:
            x = synth.act_normal(M, K, seed=seed * 10 + M)
            run_w4a16(x, wref, K, nv.OUT_BF16, n_rows=cols)


def test_w4a16_zero_rows():
    wref = oracle_weight(synth.weight_normal(64, 256, seed=4))
    x = np.zeros((3, 256), np.uint16)
    W = dev_weight(wref, 256)
    y = nv.nvfp4_gemm_w4a16(to_dev(x), W, nv.OUT_F32)
    assert float(y.abs().max()) == 0.0
    y0 = nv.nvfp4_gemm_w4a16(to_dev(np.zeros((0, 256), np.uint16)), W)
    assert y0.shape == (0, 64)


# ------------------------------------------------------------------ W4A4 ---

@pytest.mark.parametrize("shape", [(256, 256), (200, 320), (300, 512), (520, 1024)])
@pytest.mark.parametrize("M", [1, 5, 128, 130])
def test_w4a4_small(shape, M):
    N, K = shape
    wref = oracle_weight(synth.weight_normal(N, K, seed=N * 3 + K, outlier_frac=0.01))
    x = synth.act_student_t(M, K, seed=M + 1000)
    run_w4a4(x, wref, K, nv.OUT_F32)
    run_w4a4(x, wref, K, nv.OUT_BF16)


@pytest.mark.parametrize("N", [9768, 19528])
@pytest.mark.parametrize("M", [1, 37, 128])
def test_w4a4_narrow_tiles_ragged(N, M):
    """M <= 128 runs one CTA per weight tile with the narrowest tile (64, 128
    or 256 rows) whose tiles fit one wave; on a 152-SM GB300 these N take 128-
    and 256-row tiles, each with a partial last tile (40 and 72 rows; the
    256-row one has no rows in its second 128-row scale tile)."""
    K = 256
    wref = oracle_weight(synth.weight_normal(N, K, seed=N + 7, outlier_frac=0.01))
    x = synth.act_student_t(M, K, seed=M + 3000)
    run_w4a4(x, wref, K, nv.OUT_F32)
    run_w4a4(x, wref, K, nv.OUT_BF16)
    assert nv.nvfp4_get_device_status() == 0


def each_w4a4_kernel(fn):
    """Runs fn() with each W4A4 kernel for M > 128 forced in turn: CTA pairs,
    single CTAs (M <= 128 has one kernel)."""
    saved = nv.nvfp4_get_w4a4_cluster()
    try:
        for ctas in (2, 1):
            nv.nvfp4_set_w4a4_cluster(ctas)
            fn()
    finally:
        nv.nvfp4_set_w4a4_cluster(saved)


@pytest.mark.parametrize("shape", [(256, 256), (200, 320), (300, 512), (520, 1024), (1000, 4160)])
@pytest.mark.parametrize("M", [129, 160, 200, 256, 300, 513])
def test_w4a4_both_kernels(shape, M):
    """Every W4A4 kernel for M > 128 matches the oracle: ragged M (a CTA pair
    whose second CTA has no rows), ragged N (a tile whose second weight half
    is empty or partial, an odd number of 256-wide tiles), K with a partial
    last stage."""
    N, K = shape
    wref = oracle_weight(synth.weight_normal(N, K, seed=N * 5 + K, outlier_frac=0.01))
    x = synth.act_student_t(M, K, seed=M + 2000)

    def check():
        run_w4a4(x, wref, K, nv.OUT_F32)
        run_w4a4(x, wref, K, nv.OUT_BF16)
    each_w4a4_kernel(check)
    assert nv.nvfp4_get_device_status() == 0


def test_w4a4_prefill_shapes():
    wref = oracle_weight(synth.prefill_weight())
    cols = sample_rows(11008, 256, 2)
    for M in synth.PREFILL_M:
        x = synth.prefill_act(M)
        rows = None if M <= 256 else sample_rows(M, 64, M)
        worst = run_w4a4(x, wref, 4096, nv.OUT_BF16, m_rows=rows, n_rows=cols)
        print(f"prefill M={M}: worst normwise rel err {worst:.2e}")


def test_fp4_mma_rate_measurement():
    """The FP4 MMA-rate measurement behind the W4A4 roofline denominator runs
    to completion on every CTA pair (no bounded wait runs out) and reports a
    plausible rate and clock."""
    r = nv.nvfp4_measure_fp4_mma(500)
    assert nv.nvfp4_get_device_status() == nv.OK
    assert r["pairs"] >= 1 and r["tflops"] > 0, r
    assert 300 < r["sm_mhz"] < 3000, r


@pytest.mark.parametrize("shape", [(200, 16), (64, 48), (130, 80), (257, 1040), (96, 16 * 129)])
@pytest.mark.parametrize("M", [1, 7, 9, 64])
def test_w4a16_k_multiple_of_16(shape, M):
    """Weights whose K is a multiple of 16 but not of 64 (K = 16 x odd
    included, rows of 8 x odd code bytes): W4A16 through the plain kernel,
    both output types, against the oracle; the linear call takes W4A16 for
    them at any M."""
    N, K = shape
    wref = oracle_weight(synth.weight_normal(N, K, seed=N + 5 * K, outlier_frac=0.01))
    x = synth.act_normal(M, K, seed=70 + M)
    run_w4a16(x, wref, K, nv.OUT_F32)
    run_w4a16(x, wref, K, nv.OUT_BF16)
    W = dev_weight(wref, K)
    y = nv.nvfp4_linear(to_dev(x), W, nv.OUT_F32)
    assert torch.equal(y, nv.nvfp4_gemm_w4a16(to_dev(x), W, nv.OUT_F32))
    assert nv.nvfp4_get_device_status() == 0
