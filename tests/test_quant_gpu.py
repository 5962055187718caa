"""Quantisers on the GPU against the CPU oracle: bit-exact codes, scales
(logical and MMA tiling), M=4/M=6 choices, M=4 counts and tensor scales."""
import os

import numpy as np
import pytest

import oracle
import synth
from nvfp4_testutil import THREADS, to_dev, to_np_u8

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import nvfp4_weight_quantized_gb300 as nv  # noqa: E402

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from nvfp4_weight_quantized_gb300 import build
    build.build()
    nv.lib()


def _f32_bits(v):
    return np.float32(v).view(np.uint32)


def check_fos(w_bits, divisor=None):
    K = w_bits.shape[1]
    q = nv.nvfp4_quantize_fos(to_dev(w_bits), 0.0 if divisor is None else divisor)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_device_status() == nv.OK
    ts = oracle.tensor_scale(w_bits, oracle.DEFAULT_DIVISOR if divisor is None else divisor)
    ref = oracle.quantize_rows(w_bits, ts, True, THREADS)
    assert _f32_bits(q.tensor_scale.item()) == _f32_bits(ts)
    np.testing.assert_array_equal(to_np_u8(q.codes), ref["codes"])
    np.testing.assert_array_equal(to_np_u8(q.scales), ref["scales"])
    np.testing.assert_array_equal(to_np_u8(q.choice), ref["choice"])
    np.testing.assert_array_equal(to_np_u8(q.scales_mma), oracle.scales_to_mma(ref["scales"], K))
    assert int(q.m4_count.item()) == ref["m4_count"]
    return ref


def check_act(x_bits):
    K = x_bits.shape[1]
    q = nv.nvfp4_quantize_act(to_dev(x_bits), logical_scales=True)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_device_status() == nv.OK
    ts = oracle.tensor_scale(x_bits)
    ref = oracle.quantize_rows(x_bits, ts, False, THREADS)
    assert _f32_bits(q.tensor_scale.item()) == _f32_bits(ts)
    np.testing.assert_array_equal(to_np_u8(q.codes), ref["codes"])
    np.testing.assert_array_equal(to_np_u8(q.scales), ref["scales"])
    np.testing.assert_array_equal(to_np_u8(q.scales_mma), oracle.scales_to_mma(ref["scales"], K))
    return ref


def test_tiny_case():
    w, _ = synth.tiny_case()
    ref = check_fos(w)
    assert 0 < ref["m4_count"] < ref["choice"].size


def test_decode_weight_4096x4096():
    ref = check_fos(synth.decode_weight())
    print(f"decode weight: M=4 fraction {ref['m4_count'] / ref['choice'].size:.4f}")


def test_mlp_weights():
    gate_up, down = synth.mlp_weights()
    for name, w in (("gate_up", gate_up), ("down", down)):
        ref = check_fos(w)
        print(f"{name}: M=4 fraction {ref['m4_count'] / ref['choice'].size:.4f}")


@pytest.mark.parametrize("which", range(4), ids=[s[0] for s in synth.MODEL_LAYER_SHAPES])
def test_model_layer0(which):
    check_fos(synth.model_layer_weight(0, which))


@pytest.mark.parametrize("shape", [(1, 16), (3, 48), (129, 80), (300, 1040), (7, 4112), (2, 16 * 1031)])
def test_ragged_shapes(shape):
    N, K = shape
    check_fos(synth.weight_normal(N, K, seed=N * 7 + K, outlier_frac=0.02))
    check_act(synth.act_student_t(N, K, seed=N * 11 + K))


def test_fos_on_activations():
    """FourOverSix applied to activation-shaped tensors (Student-t tokens, the
    prefill distribution), the activation option of nvfp4_linear: codes,
    scales, choices and tensor scale bit-exact against the oracle."""
    for M, K, seed in ((130, 1024, 3), (257, 4096, 4)):
        check_fos(synth.act_student_t(M, K, seed=seed))


def test_custom_divisor():
    w = synth.weight_normal(64, 512, seed=77, outlier_frac=0.02)
    check_fos(w, divisor=4 * 448.0)
    check_fos(w, divisor=1000.0)


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([c.strip() for c in line.split("|")])
    return rows


def test_worked_examples_on_gpu():
    """Every hand-computed block with ts = 1 inside one tensor (an extra block
    holding 2688 = 6 * 448 makes the tensor scale exactly 1)."""
    rows = [r for r in _golden_rows("fos_worked_examples.txt") if float(r[1]) == 1.0]
    vals = [[float(v) for v in r[2].split()] for r in rows] + [[2688.0] + [0.0] * 15]
    w = synth.f32_to_bf16_bits(np.array(vals, np.float32).reshape(1, -1))
    assert (synth.bf16_bits_to_f32(w).reshape(-1, 16) == np.array(vals, np.float32)).all()
    check_fos(w)
    q = nv.nvfp4_quantize_fos(to_dev(w))
    codes, scales, choice = to_np_u8(q.codes)[0], to_np_u8(q.scales)[0], to_np_u8(q.choice)[0]
    for b, r in enumerate(rows):
        assert scales[b] == int(r[8], 16), r[0]
        assert choice[b] == int(r[7]), r[0]
        assert list(codes[8 * b:8 * b + 8]) == [int(x, 16) for x in r[9].split()], r[0]


def test_exact_ties_on_the_e2m1_grid():
    """With ts = 1 and power-of-two block scales every E2M1 midpoint is hit
    exactly, which exercises round-half-to-even in the hardware conversion."""
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    blocks = []
    for e in range(-6, 7):  # block amax 6 * 2^e -> s6 = 2^e exactly
        s = 2.0 ** e
        blk = [6 * s] + [m * s for m in mids] + [-m * s for m in mids] + [0.0]
        blocks.append(blk)
    blocks.append([2688.0] + [0.0] * 15)
    w = synth.f32_to_bf16_bits(np.array(blocks, np.float32).reshape(1, -1))
    check_fos(w)
    x = synth.f32_to_bf16_bits(np.array(blocks, np.float32).reshape(2, -1))
    check_act(x)


def test_block_scale_ties_on_the_e4m3_grid():
    """Blocks whose amax / 6 / ts is exactly an E4M3 rounding midpoint (and
    one bf16 step either side), with ts a power of two: the M=6 scale must
    round ties to even exactly as the oracle's binary32 steps do."""
    vals = []
    for e in range(-6, 9):          # normal E4M3 binades 2^-6 .. 2^8
        for m in range(8):
            lo = 2.0 ** e * (1 + m / 8)
            hi = 2.0 ** e * (1 + (m + 1) / 8)
            if hi <= 448:
                vals.append((lo + hi) / 2)
    for m in range(1, 8):           # subnormal steps m * 2^-9
        vals.append((m + 0.5) * 2.0 ** -9)
    ts = 2.0 ** -5
    amax = 2688 * ts                # tensor scale exactly ts
    blocks = []
    for v in vals:
        b = np.float32(6 * v * ts)
        for delta in (-1, 0, 1):    # one bf16 step below / at / above the midpoint
            bits = synth.f32_to_bf16_bits(np.array([b], np.float32))[0].astype(np.int64) + delta
            blk = np.zeros(16, np.uint16)
            blk[0] = np.uint16(bits)
            blk[5] = synth.f32_to_bf16_bits(np.array([b * np.float32(0.3)], np.float32))[0]
            blocks.append(blk)
    head = np.zeros(16, np.uint16)
    head[0] = synth.f32_to_bf16_bits(np.array([amax], np.float32))[0]
    blocks.append(head)
    rows = (len(blocks) + 7) // 8
    while len(blocks) < rows * 8:
        blocks.append(np.zeros(16, np.uint16))
    w = np.stack(blocks).reshape(rows, 8 * 16)
    check_fos(w)


def _blocks_to_rows(blocks, per_row=64):
    """Blocks [n, 16] of bf16 bits laid out as rows of per_row blocks (zero
    blocks pad the last row)."""
    rows = -(-len(blocks) // per_row)
    pad = np.zeros((rows * per_row - len(blocks), 16), np.uint16)
    return np.concatenate([blocks, pad]).reshape(rows, per_row * 16)


def every_bf16_below_block_max():
    """Every finite bf16 value of magnitude <= 6, both signs, 15 to a block
    behind a 6; one leading block holds 2688 so that the tensor scale is 1."""
    pos = np.arange(0, 0x40C0 + 1, dtype=np.uint16)  # +0 .. 6.0
    vals = np.concatenate([pos, pos | np.uint16(0x8000)])
    n = -(-len(vals) // 15)
    vals = np.concatenate([vals, np.zeros(n * 15 - len(vals), np.uint16)])
    blocks = np.zeros((n + 1, 16), np.uint16)
    blocks[0, 0] = 0x4528  # 2688
    blocks[1:, 0] = 0x40C0  # 6.0
    blocks[1:, 1:] = vals.reshape(n, 15)
    return _blocks_to_rows(blocks)


def every_bf16_as_block_max():
    """Every positive finite bf16 value up to 2688 as the maximum of its own
    block, beside a partner of 0.3 times it; 2688 itself makes ts = 1."""
    v = np.arange(1, 0x4528 + 1, dtype=np.uint16)
    partner = synth.f32_to_bf16_bits((synth.bf16_bits_to_f32(v) * np.float32(0.3)).astype(np.float32))
    blocks = np.zeros((len(v), 16), np.uint16)
    blocks[:, 0] = v
    blocks[:, 7] = partner
    return _blocks_to_rows(blocks)


def test_every_bf16_value_below_the_block_max():
    """With ts = 1 and block maximum 6 the M=6 candidate divides by 1 and the
    M=4 candidate by 1.5: every finite bf16 input of magnitude <= 6 goes
    through both E2M1 roundings, in the weight and the activation quantiser."""
    w = every_bf16_below_block_max()
    assert check_fos(w)["ts"] == 1.0
    check_act(w)


def test_every_bf16_value_as_a_block_max():
    """Every M=6 scale E4M3(v / 6) for v over all positive finite bf16 values
    up to 2688 (subnormal scales to 448), and the M=4 scale derived from it."""
    w = every_bf16_as_block_max()
    assert check_fos(w)["ts"] == 1.0
    check_act(w)


def test_zero_and_negative_zero():
    z = np.zeros((4, 64), np.uint16)
    z[1, 5] = 0x8000
    z[3, 63] = 0x8000
    ref = check_fos(z)
    assert ref["ts"] == 1.0


def test_nonfinite_input_sets_device_status():
    w = synth.weight_normal(32, 64, seed=3)
    w[7, 9] = 0x7F80  # +inf
    W = to_dev(w)
    nv.nvfp4_quantize_fos(W)
    assert nv.nvfp4_get_device_status() == nv.ERR_NONFINITE
    assert nv.nvfp4_get_device_status() == nv.OK  # reading clears it
    w[7, 9] = 0xFFC1  # NaN
    nv.nvfp4_quantize_act(to_dev(w))
    assert nv.nvfp4_get_device_status() == nv.ERR_NONFINITE


def test_activation_quantiser_prefill_shapes():
    for M in (64, 256, 1024):
        check_act(synth.prefill_act(M))


@pytest.mark.parametrize("shape", [(1, 16), (129, 80), (300, 1040), (4096, 4096), (5000, 2048)])
def test_both_launch_forms(shape):
    """The single-launch quantiser (tiles kept in shared memory across the
    grid-wide barrier, the rest read again) and the two-launch form (the
    default) give the same bits, both against the oracle: small tensors, a tensor with more
    tiles per CTA than stay resident, a ragged row count; FourOverSix and
    activations; and the non-finite status in both."""
    N, K = shape
    w = synth.weight_normal(N, K, seed=N + 13 * K, outlier_frac=0.01)
    saved = nv.nvfp4_get_single_launch_quantizer()
    try:
        outs = []
        for single in (True, False):
            nv.nvfp4_set_single_launch_quantizer(single)
            check_fos(w)
            if N * K <= 300 * 1040:
                check_act(synth.act_student_t(N, K, seed=N + K))
            q = nv.nvfp4_quantize_fos(to_dev(w))
            outs.append([to_np_u8(t) for t in (q.codes, q.scales, q.scales_mma, q.choice)] + [q.tensor_scale.item()])
            bad = w.copy()
            bad[N // 2, K // 3] = 0x7FC0  # NaN
            nv.nvfp4_quantize_fos(to_dev(bad))
            assert nv.nvfp4_get_device_status() == nv.ERR_NONFINITE
        for a, b in zip(outs[0], outs[1]):
            assert np.array_equal(a, b)
    finally:
        nv.nvfp4_set_single_launch_quantizer(saved)
