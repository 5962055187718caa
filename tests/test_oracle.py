"""Pins for the CPU oracle (no GPU).

Each test ties the oracle to something other than itself: the value set the
pages print, hand-computed worked examples, a third-party implementation of
the number formats (ml_dtypes), a plain library matmul, brute-force search over
every E4M3 scale, and invariants of the FourOverSix rule.
"""
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([c.strip() for c in line.split("|")])
    return rows


# ------------------------------------------------------------------ formats ---

def test_e2m1_value_set_matches_page():
    with open(os.path.join(GOLDEN, "e2m1_value_set.txt")) as f:
        printed = [float(v) for line in f if not line.startswith("#") for v in line.split()]
    decoded = [oracle.e2m1_value(c) for c in range(16)]
    assert sorted(set(decoded)) == sorted(set(printed))
    assert max(abs(v) for v in decoded) == 6.0
    # +0 and -0 are the only pair of codes with equal value
    assert len(set(decoded)) == 15
    assert np.signbit(oracle.e2m1_value(8)) and not np.signbit(oracle.e2m1_value(0))
    # codes 0..7 are the positive magnitudes in increasing order, 8..15 their negatives
    assert decoded[:8] == sorted(decoded[:8])
    assert all(decoded[c + 8] == -decoded[c] for c in range(8))


def test_e2m1_round_to_nearest_even_and_saturate():
    # midpoints go to the neighbour whose code is even
    table = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for v, want in table.items():
        assert oracle.e2m1_value(oracle.e2m1_encode(v)) == want
        assert oracle.e2m1_value(oracle.e2m1_encode(-v)) == -want
    for v in (6.0, 6.5, 7.0, 100.0, 3e38, float("inf")):
        assert oracle.e2m1_encode(v) == 7
        assert oracle.e2m1_encode(-v) == 15
    assert oracle.e2m1_encode(-0.1) == 8  # negative values rounding to 0 keep the sign
    assert oracle.e2m1_encode(0.0) == 0 and oracle.e2m1_encode(-0.0) == 8
    for c in range(16):  # every grid value round-trips
        assert oracle.e2m1_encode(oracle.e2m1_value(c)) == c


def test_e2m1_encode_matches_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    rng = np.random.default_rng(7)
    vals = np.concatenate([np.arange(-8, 8, 1 / 64, dtype=np.float32),
                           rng.standard_normal(4000).astype(np.float32) * 3,
                           np.nextafter(np.float32([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]), 0),
                           np.nextafter(np.float32([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]), 9)])
    lib = vals.astype(ml.float4_e2m1fn).view(np.uint8) & 0xF
    mine = np.array([oracle.e2m1_encode(float(v)) for v in vals], np.uint8)
    np.testing.assert_array_equal(mine, lib)


def test_e4m3_decode_matches_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    lib = np.arange(256, dtype=np.uint8).view(ml.float8_e4m3fn).astype(np.float64)
    mine = np.array([oracle.e4m3_value(b) for b in range(256)])
    np.testing.assert_array_equal(np.isnan(mine), np.isnan(lib))
    ok = ~np.isnan(lib)
    np.testing.assert_array_equal(mine[ok], lib[ok])
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(0x01) == 2.0 ** -9


def test_e4m3_encode_matches_ml_dtypes_in_range():
    ml = pytest.importorskip("ml_dtypes")
    pos = np.arange(127, dtype=np.uint8).view(ml.float8_e4m3fn).astype(np.float64)
    mids = (pos[:-1] + pos[1:]) / 2
    rng = np.random.default_rng(3)
    vals = np.concatenate([pos, mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9),
                           rng.uniform(0, 460, 20000), 2.0 ** rng.uniform(-14, 8.8, 20000)])
    vals = vals.astype(np.float32)
    vals = vals[vals < 464]  # beyond 464 ml_dtypes produces NaN; saturation is tested below
    lib = vals.astype(ml.float8_e4m3fn).view(np.uint8)
    mine = np.array([oracle.e4m3_encode(float(v)) for v in vals], np.uint8)
    np.testing.assert_array_equal(mine, lib)


def test_e4m3_saturates_to_448():
    for v in (448.0, 449.0, 464.0, 480.0, 1e6, float("inf")):
        assert oracle.e4m3_encode(v) == 0x7E


# ------------------------------------------------------- the 1.5x relation ---

def test_m4_scale_is_fp8_of_m6_times_1p5_for_every_scale():
    ml = pytest.importorskip("ml_dtypes")
    for s6 in range(1, 127):
        v = np.float32(oracle.e4m3_value(s6)) * np.float32(1.5)  # exact in binary32
        assert float(v) == oracle.e4m3_value(s6) * 1.5
        s4 = oracle.e4m3_encode(float(v))
        if v < 464:
            assert s4 == int(np.float32(v).astype(ml.float8_e4m3fn).view(np.uint8))
        else:
            assert s4 == 0x7E
        # "about 1.5x": for normal E4M3 values the re-rounding moves the product by
        # at most half a mantissa step (1/16 relative) unless it saturates
        if oracle.e4m3_value(s6) >= 2.0 ** -6 and oracle.e4m3_value(s6) * 1.5 <= 448:
            assert abs(oracle.e4m3_value(s4) / (oracle.e4m3_value(s6) * 1.5) - 1) <= 0.0625


# ------------------------------------------------------- worked examples ---

@pytest.mark.parametrize("row", _golden_rows("fos_worked_examples.txt"), ids=lambda r: r[0])
def test_fos_worked_example(row):
    name, ts, vals, s6, s4, sse6, sse4, choice, scale, code_bytes = row
    x = np.array([float(v) for v in vals.split()], np.float32)
    r = oracle.fos_block(x, float(ts))
    assert r["s6"] == int(s6, 16), name
    assert r["s4"] == int(s4, 16), name
    assert r["sse6"] == float(sse6), name
    assert r["sse4"] == float(sse4), name
    assert r["choice"] == int(choice), name
    assert r["scale"] == int(scale, 16), name
    packed = [int(r["codes"][2 * j]) | (int(r["codes"][2 * j + 1]) << 4) for j in range(8)]
    assert packed == [int(b, 16) for b in code_bytes.split()], name


@pytest.mark.parametrize("row", _golden_rows("sse_tree_order.txt"), ids=lambda r: r[0])
def test_sse_tree_order(row):
    name, sbyte, ts, vals, sse = row
    x = np.array([float(v) for v in vals.split()], np.float32)
    got, _ = oracle.block_sse(x, int(sbyte, 16), float(ts))
    assert got == float(np.float32(float(sse))), name


def test_worked_examples_through_whole_tensor_path():
    """The m4_wins / grid_m6_exact blocks inside a tensor whose amax gives ts = 1
    exactly (amax 2688 = 6 * 448 is a bf16 value)."""
    rows = {r[0]: r for r in _golden_rows("fos_worked_examples.txt")}
    blocks = []
    for name in ("grid_m6_exact", "m4_wins", "tie_keeps_m6"):
        blocks.append([float(v) for v in rows[name][2].split()])
    blocks.append([2688.0] + [0.0] * 15)
    w = synth.f32_to_bf16_bits(np.array(blocks, np.float32).reshape(1, -1))
    q = oracle.quantize_fos(w)
    assert q["ts"] == 1.0
    assert list(q["choice"][0]) == [0, 1, 0, 0]
    assert list(q["scales"][0][:3]) == [0x38, 0x3C, 0x38]
    assert q["m4_count"] == 1
    assert list(q["codes"][0][8:16]) == [0x56, 0x24, 0x01, 0xDE, 0xAC, 0x09, 0x56, 0x24]


# --------------------------------------------------------------- invariants ---

def _random_blocks(n, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, 16)).astype(np.float32)
    x *= np.exp(rng.uniform(-3, 3, (n, 1))).astype(np.float32)
    mask = rng.random((n, 16)) < 0.05
    x[mask] *= 8
    return x


def test_selection_rule_invariants():
    x = _random_blocks(3000, 11)
    ts = float(np.abs(x).max() / 2688.0)
    m4 = 0
    for blk in x:
        r = oracle.fos_block(blk, ts)
        assert r["choice"] == int(r["sse4"] < r["sse6"])
        chosen = r["s4"] if r["choice"] else r["s6"]
        assert r["scale"] == chosen
        sse, q = oracle.block_sse(blk, chosen, ts)
        assert sse == min(r["sse4"], r["sse6"])
        np.testing.assert_array_equal(q, r["codes"])
        m4 += r["choice"]
    assert 0 < m4 < len(x)  # both choices occur on generic data


def test_no_magnitude_six_code_in_unsaturated_m4_blocks():
    """x / eff4 <= 4 (1 + 2^-4)^2 < 5 when s6 is a normal E4M3 value and s4 is not
    saturated, so an M=4 block never uses the code for 6."""
    x = _random_blocks(3000, 12)
    ts = float(np.abs(x).max() / 2688.0)
    seen = 0
    for blk in x:
        r = oracle.fos_block(blk, ts)
        if r["choice"] and oracle.e4m3_value(r["s6"]) >= 2.0 ** -6 and r["s4"] != 0x7E:
            seen += 1
            assert not np.any((r["codes"] & 7) == 7)
    assert seen > 100


def test_constant_and_zero_blocks():
    # a constant block c with |c|/6 an E4M3 value is exact under both candidates
    # (|c| -> 6 * s6 and, with s4 = 1.5 * s6, -> 4 * s4), so the tie keeps M=6
    for c in (6.0, -3.0, 0.75):
        r = oracle.fos_block(np.full(16, c, np.float32), 1.0)
        assert oracle.e4m3_value(r["s6"]) == abs(c) / 6
        assert oracle.e4m3_value(r["s4"]) == 1.5 * abs(c) / 6
        assert r["sse6"] == 0.0 and r["sse4"] == 0.0 and r["choice"] == 0
        assert np.all(r["codes"] == (15 if c < 0 else 7))
    r = oracle.fos_block(np.zeros(16, np.float32), 0.01)
    assert r["scale"] == 0 and r["choice"] == 0 and not r["codes"].any()


# --------------------------------------------------------------- brute force ---

def _grid_nearest_sse(x64, eff):
    """Exact (binary64) SSE of the block when every element takes the nearest
    of the 15 E2M1 grid values times eff (exhaustive search)."""
    grid = np.array(sorted({oracle.e2m1_value(c) for c in range(16)}))
    if eff == 0:
        return float(np.sum(x64 ** 2))
    cand = grid[None, :] * eff
    d = np.min(np.abs(x64[:, None] - cand), axis=1)
    return float(np.sum(d ** 2))


def test_brute_force_scale_search_on_tiny_blocks():
    ml = pytest.importorskip("ml_dtypes")
    e4 = np.arange(127, dtype=np.uint8).view(ml.float8_e4m3fn).astype(np.float64)
    x = _random_blocks(400, 13)
    ts = float(np.float32(np.abs(x).max() / 2688.0))
    for blk in x:
        r = oracle.fos_block(blk, ts)
        x64 = blk.astype(np.float64)
        amax = float(np.float32(np.abs(blk).max()))
        r6 = float(np.float32(np.float32(amax / np.float32(6)) / np.float32(ts)))
        # (i) s6 is the E4M3 value nearest r6
        dist = np.abs(e4 - r6)
        assert dist[r["s6"]] == dist.min()
        # (ii) the oracle's SSEs agree with exhaustive nearest-grid evaluation
        b6 = _grid_nearest_sse(x64, e4[r["s6"]] * np.float64(np.float32(ts)))
        b4 = _grid_nearest_sse(x64, e4[r["s4"]] * np.float64(np.float32(ts)))
        tol = 1e-5 * max(b6, b4) + 1e-30
        assert abs(r["sse6"] - b6) <= tol and abs(r["sse4"] - b4) <= tol
        if abs(b4 - b6) > 2 * tol:
            assert r["choice"] == int(b4 < b6)
        # (iii) best over all 127 scales <= FourOverSix <= plain M=6
        best = min(_grid_nearest_sse(x64, e * np.float64(np.float32(ts))) for e in e4)
        fos = min(b4, b6)
        assert best <= fos + tol and fos <= b6 + tol


# ------------------------------------------------------------ whole tensors ---

def test_quantize_fos_matches_blockwise_and_tensor_scale():
    w = synth.weight_normal(8, 64, seed=5, outlier_frac=0.05)
    q = oracle.quantize_fos(w)
    wf = synth.bf16_bits_to_f32(w)
    assert q["ts"] == float(np.float32(np.abs(wf).max()) / np.float32(2688.0))
    for n in range(8):
        for b in range(4):
            r = oracle.fos_block(wf[n, 16 * b:16 * b + 16], q["ts"])
            assert q["scales"][n, b] == r["scale"] and q["choice"][n, b] == r["choice"]
            packed = [int(r["codes"][2 * j]) | (int(r["codes"][2 * j + 1]) << 4) for j in range(8)]
            assert list(q["codes"][n, 8 * b:8 * b + 8]) == packed
    assert q["m4_count"] == int(q["choice"].sum())


def test_quantize_zero_tensor_and_nonfinite():
    z = np.zeros((2, 32), np.uint16)
    z[0, 3] = 0x8000  # -0
    q = oracle.quantize_fos(z)
    assert q["ts"] == 1.0 and not q["scales"].any() and not q["choice"].any()
    assert q["codes"][0, 1] == 0x80 and q["codes"].sum() == 0x80
    bad = np.zeros((1, 16), np.uint16)
    bad[0, 5] = 0x7F80  # +inf
    with pytest.raises(oracle.OracleError) as e:
        oracle.quantize_fos(bad)
    assert e.value.status == 5
    bad[0, 5] = 0x7FC1  # NaN
    with pytest.raises(oracle.OracleError):
        oracle.quantize_act(bad)


def test_custom_divisor_avoids_saturation():
    """Under D = 6*448 the block holding amax gets s6 = 448, so its M=4 candidate
    saturates to 448 as well (a tie, so M=6).  Under D = 4*448 that block's s6 is
    about 299 and its s4 (about 1.5x) stays a distinct, unsaturated value."""
    w = synth.weight_normal(4, 256, seed=9, outlier_frac=0.02)
    wf = synth.bf16_bits_to_f32(w)
    n, k = np.unravel_index(np.argmax(np.abs(wf)), wf.shape)
    blk = wf[n, 16 * (k // 16):16 * (k // 16) + 16]
    a = oracle.quantize_fos(w)
    ra = oracle.fos_block(blk, a["ts"])
    assert ra["s6"] == 0x7E and ra["s4"] == 0x7E and ra["choice"] == 0
    b = oracle.quantize_fos(w, divisor=4 * 448.0)
    assert b["ts"] == float(np.float32(np.abs(wf).max()) / np.float32(1792.0))
    rb = oracle.fos_block(blk, b["ts"])
    assert oracle.e4m3_value(rb["s6"]) == 288.0 and rb["s4"] == 0x7E  # 432 ties up to 448
    assert rb["s4"] != rb["s6"]


def test_act_quant_is_m6_only():
    x = synth.act_student_t(3, 128, seed=2)
    q = oracle.quantize_act(x)
    xf = synth.bf16_bits_to_f32(x)
    for m in range(3):
        for b in range(8):
            blk = xf[m, 16 * b:16 * b + 16]
            s = oracle.fos_block(blk, q["ts"])["s6"]
            assert q["scales"][m, b] == s
            _, codes = oracle.block_sse(blk, s, q["ts"])
            packed = [int(codes[2 * j]) | (int(codes[2 * j + 1]) << 4) for j in range(8)]
            assert list(q["codes"][m, 8 * b:8 * b + 8]) == packed


def test_dequantised_weights_are_exact_in_bf16():
    """value(code) * value(scale) has at most 6 significant bits and lies in
    [2^-10, 2688], so it is exact in bfloat16 (the W4A16 kernel relies on this)."""
    for c in range(16):
        for s in range(127):
            v = np.float32(oracle.e2m1_value(c) * oracle.e4m3_value(s))
            b = synth.f32_to_bf16_bits(np.array([v]))
            assert synth.bf16_bits_to_f32(b)[0] == v


# ------------------------------------------------------------- scale layout ---

def test_scales_to_mma_layout_hand_examples():
    R, K = 130, 80  # 2 row tiles x 2 column tiles (5 blocks, padded to 8)
    s = np.arange(R * (K // 16), dtype=np.uint32).reshape(R, K // 16)
    s = (s % 251 + 1).astype(np.uint8)
    out = oracle.scales_to_mma(s, K)
    assert out.size == 2 * 2 * 512
    assert out[0] == s[0, 0]
    assert out[22] == s[33, 2]      # (33 % 32) * 16 + (33 // 32) * 4 + 2
    assert out[511] == s[127, 3]    # 31 * 16 + 3 * 4 + 3
    assert out[592] == s[5, 4]      # tile 1: 512 + 5 * 16
    assert out[1552] == s[129, 4]   # tile 3: 1536 + 1 * 16
    # every logical scale appears exactly once; padding is zero
    assert np.count_nonzero(out) == R * (K // 16)
    assert sorted(out[out > 0].tolist()) == sorted(s.ravel().tolist())


# -------------------------------------------------------------------- GEMMs ---

def _dequant_lib(codes, scales, ts):
    ml = pytest.importorskip("ml_dtypes")
    lo = codes & 0xF
    hi = codes >> 4
    nib = np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1)
    v = nib.astype(np.uint8).view(ml.float4_e2m1fn).astype(np.float64)
    s = scales.view(ml.float8_e4m3fn).astype(np.float64)
    return v * np.repeat(s, 16, axis=1) * np.float64(ts)


def test_gemm_w4a16_by_hand():
    x = synth.f32_to_bf16_bits(np.array([[1.0, 2.0] + [0.0] * 14], np.float32))
    codes = np.zeros((1, 8), np.uint8)
    codes[0, 0] = 0x7 | (0xA << 4)  # element 0 -> 6, element 1 -> -1
    scales = np.array([[0x38]], np.uint8)  # 1.0
    y = oracle.gemm_w4a16(x, codes, scales, 0.5)
    assert y[0, 0] == 1 * 6 * 0.5 + 2 * (-1) * 0.5  # = 2


def test_gemm_w4a16_matches_library_matmul():
    w = synth.weight_normal(48, 96, seed=21, outlier_frac=0.02)
    x = synth.act_normal(5, 96, seed=22)
    q = oracle.quantize_fos(w)
    y = oracle.gemm_w4a16(x, q["codes"], q["scales"], q["ts"])
    ref = synth.bf16_bits_to_f32(x).astype(np.float64) @ _dequant_lib(q["codes"], q["scales"], q["ts"]).T
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    rows = oracle.gemm_w4a16_rows(x, [4, 1], q["codes"], q["scales"], q["ts"])
    np.testing.assert_array_equal(rows, y[[4, 1]])


def test_gemm_w4a4_matches_library_matmul():
    w = synth.weight_normal(40, 64, seed=23, outlier_frac=0.02)
    x = synth.act_student_t(6, 64, seed=24)
    qw = oracle.quantize_fos(w)
    qa = oracle.quantize_act(x)
    y = oracle.gemm_w4a4(qa["codes"], qa["scales"], qa["ts"], qw["codes"], qw["scales"], qw["ts"])
    ref = _dequant_lib(qa["codes"], qa["scales"], qa["ts"]) @ \
        _dequant_lib(qw["codes"], qw["scales"], qw["ts"]).T
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_fos_error_never_worse_than_m6_on_a_tensor():
    w = synth.weight_lognormal_rows(16, 256, seed=31)
    q = oracle.quantize_fos(w)
    wf = synth.bf16_bits_to_f32(w).astype(np.float64)
    deq = _dequant_lib(q["codes"], q["scales"], q["ts"])
    # an all-M6 quantisation of the same tensor
    ts = q["ts"]
    sse_fos = sse_m6 = 0.0
    for n in range(16):
        for b in range(16):
            blk = wf[n, 16 * b:16 * b + 16].astype(np.float32)
            r = oracle.fos_block(blk, ts)
            sse_fos += min(r["sse4"], r["sse6"])
            sse_m6 += r["sse6"]
    assert sse_fos <= sse_m6
    assert np.sum((wf - deq) ** 2) == pytest.approx(sse_fos, rel=1e-5)


# ------------------------------------------- dequantisation and QAT backward ---

# E2M1 magnitudes as the pages print them (codes 0..7); sign bit 3
_E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _e4m3(byte: int) -> float:
    """E4M3 by its definition (bias 7, subnormals 0.m * 2^-6)."""
    e, m = (byte >> 3) & 15, byte & 7
    return (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)


def _exact_dequant(codes, scales, ts):
    R, K = codes.shape[0], codes.shape[1] * 2
    out = np.zeros((R, K))
    for r in range(R):
        for k in range(K):
            c = (codes[r, k // 2] >> (4 * (k & 1))) & 15
            v = _E2M1[c & 7] * (-1.0 if c & 8 else 1.0)
            out[r, k] = v * _e4m3(int(scales[r, k // 16])) * ts
    return out


def test_dequant_bf16_exact_when_representable():
    """With ts a power of two every value(code) * value(scale) * ts has at
    most 6 significant bits, so its bf16 is exact: the oracle must return it."""
    rng = np.random.default_rng(11)
    codes = rng.integers(0, 256, size=(6, 32), dtype=np.uint8)
    scales = rng.integers(0, 0x7F, size=(6, 4), dtype=np.uint8)  # below the NaN pattern
    for ts in (1.0, 2.0 ** -10, 2.0 ** 5):
        got = synth.bf16_bits_to_f32(oracle.dequant_bf16(codes, scales, ts)).astype(np.float64)
        assert np.array_equal(got, _exact_dequant(codes, scales, ts))


def test_dequant_bf16_rounding_bound():
    """For any tensor scale the result is the exact value rounded twice
    (binary32 then bf16): within half a bf16 step plus 2^-24 relative, and
    monotone in the exact value within a row."""
    rng = np.random.default_rng(12)
    codes = rng.integers(0, 256, size=(4, 64), dtype=np.uint8)
    scales = rng.integers(0x08, 0x7F, size=(4, 8), dtype=np.uint8)
    for ts in (0.0123456789, 3.3e-5, 171.7):
        ts32 = float(np.float32(ts))
        exact = _exact_dequant(codes, scales, ts32)
        got = synth.bf16_bits_to_f32(oracle.dequant_bf16(codes, scales, ts32)).astype(np.float64)
        err = np.abs(got - exact)
        assert np.all(err <= np.abs(exact) * (2.0 ** -8 + 2.0 ** -24) + 1e-300)
        o = np.argsort(exact, axis=None, kind="stable")
        assert np.all(np.diff(got.reshape(-1)[o]) >= 0)


def test_dequant_bf16_ties_by_hand():
    """Round-to-nearest-even at both steps, worked by hand on a block with
    scale 0x38 (value 1):
    - code 2 (+1) and code 0xA (-1) times ts = 1 + 2^-8: the binary32 product
      is exact and is the midpoint of the bf16 values 1 (0x3f80) and 1 + 2^-7
      (0x3f81), so the even 0x3f80; with ts = 1 + 3 * 2^-8 the midpoint of
      0x3f81 and 0x3f82, so 0x3f82;
    - code 3 (+1.5) and 0xB (-1.5) times ts = 11228502 * 2^-24: the exact
      product is 1 + 2^-8 + 2^-24, a binary32 tie that rounds to the even
      1 + 2^-8, itself a bf16 tie, so 0x3f80 (rounding the exact product to
      bf16 in one step would give 0x3f81)."""
    scales = np.array([[0x38]], np.uint8)
    cases = [(0x02 | (0x0A << 4), 1.0 + 2.0 ** -8, 0x3F80),
             (0x02 | (0x0A << 4), 1.0 + 3 * 2.0 ** -8, 0x3F82),
             (0x03 | (0x0B << 4), 11228502 * 2.0 ** -24, 0x3F80)]
    for byte, ts, want in cases:
        assert float(np.float32(ts)) == ts
        codes = np.array([[byte] + [0] * 7], np.uint8)
        got = oracle.dequant_bf16(codes, scales, ts)[0]
        assert list(got[:2]) == [want, want | 0x8000], (hex(byte), ts)
        assert not got[2:].any()


def test_dequant_bf16_agrees_with_gemm_oracle():
    """Against the GEMM oracle's own binary64 dequantisation (unit-vector
    activations pick out W_hat): equal up to the two roundings."""
    w = synth.weight_normal(8, 64, seed=13, outlier_frac=0.05)
    q = oracle.quantize_fos(w)
    eye = synth.f32_to_bf16_bits(np.eye(64, dtype=np.float32))
    w_hat = oracle.gemm_w4a16(eye, q["codes"], q["scales"], q["ts"]).T  # [8, 64]
    got = synth.bf16_bits_to_f32(oracle.dequant_bf16(q["codes"], q["scales"], q["ts"])).astype(np.float64)
    assert np.all(np.abs(got - w_hat) <= np.abs(w_hat) * (2.0 ** -8 + 2.0 ** -24))


def test_qat_backward_brute_force():
    """dX = dY W_hat and dW = dY^T X_hat against explicit sums on a tiny case."""
    rng = np.random.default_rng(14)
    M, N, K = 3, 4, 16
    dy = synth.f32_to_bf16_bits(rng.standard_normal((M, N)).astype(np.float32))
    w = synth.f32_to_bf16_bits(rng.standard_normal((N, K)).astype(np.float32))
    x = synth.f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    dx, dw = oracle.qat_backward(dy, w, x)
    f = lambda b: synth.bf16_bits_to_f32(b).astype(np.float64)  # noqa: E731
    DY, W, X = f(dy), f(w), f(x)
    for m in range(M):
        for k in range(K):
            assert np.isclose(dx[m, k], sum(DY[m, n] * W[n, k] for n in range(N)), rtol=1e-14, atol=1e-14)
    for n in range(N):
        for k in range(K):
            assert np.isclose(dw[n, k], sum(DY[m, n] * X[m, k] for m in range(M)), rtol=1e-14, atol=1e-14)


# ------------------------------------------------------------ GPTQ + FOS ---

def _hessian(K, T, seed):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((T, K)).astype(np.float32)
    X[:, : K // 4] *= 3.0  # unequal feature scales
    return (2.0 * X.T @ X / T).astype(np.float32)


def _dequant64(codes, scales, ts):
    N, K = codes.shape[0], codes.shape[1] * 2
    e2 = np.array([oracle.e2m1_value(c) for c in range(16)])
    e4 = np.array([oracle.e4m3_value(b) if (b & 0x7F) != 0x7F else 0.0 for b in range(256)])
    q = np.stack([codes & 15, codes >> 4], axis=-1).reshape(N, K)
    return e2[q] * np.repeat(e4[scales], 16, axis=1) * ts


def test_gptq_identity_hessian_is_rtn():
    """With H = c I the inverse Hessian's Cholesky factor is diagonal, so no
    error is spread and GPTQ must return the FourOverSix round-to-nearest
    codes and scales exactly."""
    w = synth.weight_normal(48, 256, seed=21, outlier_frac=0.02)
    f = oracle.quantize_fos(w)
    for c in (1.0, 0.37):
        g = oracle.gptq_fos(w, np.eye(256, dtype=np.float32) * c, block=64)
        assert np.array_equal(g["codes"], f["codes"]) and np.array_equal(g["scales"], f["scales"])
        assert g["ts"] == f["ts"]


def test_gptq_inverse_cholesky_factor():
    """U^T U is the inverse of the damped Hessian (numpy binary64 inverse)."""
    K = 192
    H = _hessian(K, 400, 22)
    g = oracle.gptq_fos(synth.weight_normal(8, K, seed=23), H, damp=0.01, want_u=True)
    U = g["U"].astype(np.float64)
    assert np.all(np.tril(U, -1) == 0) and np.all(np.diag(U) > 0)
    Hd = H.astype(np.float64) + 0.01 * np.mean(np.diag(H.astype(np.float64))) * np.eye(K)
    inv = np.linalg.inv(Hd)
    assert np.abs(U.T @ U - inv).max() <= 1e-4 * np.abs(inv).max()


def test_gptq_lowers_layer_error():
    """GPTQ's purpose: the layer output error tr(dW H dW^T) of its codes is
    below that of round-to-nearest with the same FourOverSix scales, while
    the scales (the M=4 / M=6 choices) are unchanged."""
    K = 256
    w = synth.weight_normal(96, K, seed=24, outlier_frac=0.01)
    H = _hessian(K, 512, 25)
    f = oracle.quantize_fos(w)
    g = oracle.gptq_fos(w, H, block=64)
    assert np.array_equal(g["scales"], f["scales"])
    W = synth.bf16_bits_to_f32(w).astype(np.float64)
    H64 = H.astype(np.float64)

    def err(codes):
        d = W - _dequant64(codes, f["scales"], f["ts"])
        return float(np.einsum("nk,kl,nl->", d, H64, d))
    assert err(g["codes"]) < 0.9 * err(f["codes"])


def _code_values(codes):
    """E2M1 values of packed codes (+0 and -0 both 0)."""
    e2 = np.array([oracle.e2m1_value(c) for c in range(16)])
    return e2[np.stack([codes & 15, codes >> 4], axis=-1).reshape(codes.shape[0], -1)]


def test_gptq_ref64_pinned_to_definitions():
    """The plain binary64 GPTQ itself: with H = c I it is round-to-nearest
    under the FourOverSix scales (except where the binary32 quotient of the
    quantiser lands exactly on a rounding midpoint that the binary64 one
    misses by under 1e-6: those follow the quantiser's code), and on a small
    case each of its codes rounds the binary64 least-squares continuation of
    its row (the defining property, solved directly), away from midpoints."""
    w = synth.weight_normal(16, 128, seed=51, outlier_frac=0.02)
    f = oracle.quantize_fos(w)
    r = oracle.gptq_fos_ref64(w, np.eye(128, dtype=np.float32) * 0.5, f["scales"], f["ts"], follow=f["codes"],
                              delta=1e-6)
    assert np.array_equal(_code_values(r["codes"]), _code_values(f["codes"]))
    assert 0 < r["near"].sum() <= 0.01 * r["near"].size  # exact midpoints, and one the binary32 quotient hits
    free = oracle.gptq_fos_ref64(w, np.eye(128, dtype=np.float32) * 0.5, f["scales"], f["ts"])
    assert np.array_equal(_code_values(free["codes"])[~r["near"]], _code_values(f["codes"])[~r["near"]])
    N, K, damp = 4, 48, 0.05
    w = synth.weight_normal(N, K, seed=52, outlier_frac=0.02)
    f = oracle.quantize_fos(w)
    H = _hessian(K, 256, 53)
    r = oracle.gptq_fos_ref64(w, H, f["scales"], f["ts"], damp=damp)
    W0 = synth.bf16_bits_to_f32(w).astype(np.float64)
    H64 = H.astype(np.float64)
    Hd = H64 + damp * np.mean(np.diag(H64)) * np.eye(K)
    Q = _dequant64(r["codes"], f["scales"], f["ts"])
    e4 = np.array([oracle.e4m3_value(b) if (b & 0x7F) != 0x7F else 0.0 for b in range(256)])
    unit = np.repeat(e4[f["scales"]], 16, axis=1) * f["ts"]
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    checked = 0
    for n in range(N):
        for i in range(K):
            eF = W0[n, :i] - Q[n, :i]
            u = W0[n, i:] + (np.linalg.solve(Hd[i:, i:], Hd[i:, :i] @ eF) if i else 0.0)
            x = u[0] / unit[n, i]
            d = np.sort(np.abs(grid - abs(x)))
            if d[1] - d[0] < 1e-6:
                continue
            assert Q[n, i] / unit[n, i] == np.copysign(grid[np.argmin(np.abs(grid - abs(x)))], x), (n, i, x)
            checked += 1
    assert checked >= 0.98 * N * K


@pytest.mark.parametrize("N,K,block,damp", [(64, 512, 128, 0.01), (40, 1040, 128, 0.01), (48, 384, 48, 0.1)])
def test_gptq_binary32_oracle_agrees_with_plain_binary64(N, K, block, damp):
    """The binary32 GPTQ oracle (the GPU kernel's operation order: index
    reversal J H J, right-looking Cholesky, lazy 128-column blocks) against
    the plain unblocked binary64 GPTQ, which shares none of that order: every
    code agrees, except at elements whose binary64 quotient lies within 1e-3
    of an E2M1 rounding midpoint, where the binary64 run adopts the binary32
    code (which must be one of the two values either side) so both go on
    from the same decision.  A wrong lazy-block update or reversal changes
    the continuation by far more than rounding and fails here."""
    w = synth.weight_normal(N, K, seed=N + K, outlier_frac=0.01)
    H = _hessian(K, 2 * K, N + 7)
    g = oracle.gptq_fos(w, H, damp=damp, block=block)
    r = oracle.gptq_fos_ref64(w, H, g["scales"], g["ts"], damp=damp, follow=g["codes"], delta=1e-3)
    assert np.array_equal(_code_values(r["codes"]), _code_values(g["codes"]))
    assert r["near"].mean() < 0.01, r["near"].mean()
    assert not np.array_equal(g["codes"], oracle.quantize_fos(w)["codes"])  # errors were spread


def test_silu_mul_reference_closed_forms():
    """The binary64 silu(g) * u of the test utilities at points with closed
    forms: 0 at g = 0, the logistic value at g = 1, the limits g (g >> 0) and
    0 (g << 0, where exp overflows), the identity silu(g) - silu(-g) = g, and
    linearity in u."""
    from nvfp4_testutil import silu_mul_ref
    g = np.array([0.0, 1.0, -1.0, 40.0, -40.0, 800.0, -800.0, 2.5])
    u = np.ones_like(g)
    y = silu_mul_ref(g, u)
    assert y[0] == 0.0
    assert y[1] == pytest.approx(1.0 / (1.0 + np.exp(-1.0)), rel=1e-15)
    assert y[1] - y[2] == pytest.approx(1.0, rel=1e-15)        # silu(g) - silu(-g) = g
    assert y[3] == pytest.approx(40.0, rel=1e-15) and abs(y[4]) < 1e-15
    assert y[5] == 800.0 and y[6] == 0.0                        # exp overflow handled
    assert silu_mul_ref(np.array([2.5]), np.array([-3.0]))[0] == pytest.approx(-3.0 * y[7], rel=1e-15)


@pytest.mark.parametrize("damp,block", [(0.01, 16), (0.5, 128), (0.1, 48)])  # 48: a ragged last block
def test_gptq_codes_round_the_least_squares_continuation(damp, block):
    """GPTQ's defining property, checked without its Cholesky steps: when
    column i is quantised, the working row is the minimiser of the layer error
    (w0 - w) Hd (w0 - w)^T over the columns >= i with the columns < i held at
    their quantised values (Hd = H + damp * mean(diag H) * I).  That
    continuation is w0[i:] + Hd[i:, i:]^-1 Hd[i:, :i] (w0 - q)[:i], solved
    here in binary64 for every column; each code must be the E2M1 value
    nearest to its column under the block's fixed scale (saturating at 6).
    Elements within 1e-3 of a rounding midpoint are skipped."""
    N, K = 6, 64
    w = synth.weight_normal(N, K, seed=26, outlier_frac=0.02)
    H = _hessian(K, 1024, 27)
    g = oracle.gptq_fos(w, H, damp=damp, block=block)
    W0 = synth.bf16_bits_to_f32(w).astype(np.float64)
    H64 = H.astype(np.float64)
    Hd = H64 + damp * np.mean(np.diag(H64)) * np.eye(K)
    Q = _dequant64(g["codes"], g["scales"], g["ts"])
    e4 = np.array([oracle.e4m3_value(b) if (b & 0x7F) != 0x7F else 0.0 for b in range(256)])
    unit = np.repeat(e4[g["scales"]], 16, axis=1) * g["ts"]
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    checked = 0
    for r in range(N):
        for i in range(K):
            assert unit[r, i] > 0
            eF = W0[r, :i] - Q[r, :i]
            u = W0[r, i:] + (np.linalg.solve(Hd[i:, i:], Hd[i:, :i] @ eF) if i else 0.0)
            x = u[0] / unit[r, i]
            d = np.sort(np.abs(grid - abs(x)))
            if d[1] - d[0] < 1e-3:
                continue
            want = np.copysign(grid[np.argmin(np.abs(grid - abs(x)))], x)
            assert Q[r, i] / unit[r, i] == want, (r, i, x)
            checked += 1
    assert checked >= 0.95 * N * K
    assert not np.array_equal(g["codes"], oracle.quantize_fos(w)["codes"])  # errors were spread


def test_threaded_oracle_splits_match_single_calls():
    """The parity tests split oracle work over threads by row; every split
    (more threads than rows included) must give exactly the single-call
    result, on a ragged row count."""
    from nvfp4_testutil import oracle_w4a16, oracle_w4a4
    w = synth.weight_normal(37, 128, seed=31, outlier_frac=0.02)
    ref = oracle.quantize_fos(w)
    x = synth.act_student_t(13, 128, seed=32)
    a = oracle.quantize_act(x)
    y16 = oracle.gemm_w4a16(x, ref["codes"], ref["scales"], ref["ts"])
    y4 = oracle.gemm_w4a4(a["codes"], a["scales"], a["ts"], ref["codes"], ref["scales"], ref["ts"])
    cols = np.array([36, 0, 5, 17])
    for threads in (1, 3, 7, 64):
        q = oracle.quantize_rows(w, ref["ts"], True, threads)
        for k in ("codes", "scales", "choice"):
            assert np.array_equal(q[k], ref[k]), (k, threads)
        assert q["m4_count"] == ref["m4_count"]
        assert np.array_equal(oracle_w4a16(x, ref["codes"], ref["scales"], ref["ts"], threads=threads).y, y16)
        assert np.array_equal(oracle_w4a16(x, ref["codes"], ref["scales"], ref["ts"], n_rows=cols,
                                           threads=threads).y, y16[:, cols])
        assert np.array_equal(oracle_w4a4(a["codes"], a["scales"], a["ts"], ref["codes"], ref["scales"],
                                          ref["ts"], threads=threads).y, y4)
        assert np.array_equal(oracle_w4a4(a["codes"], a["scales"], a["ts"], ref["codes"], ref["scales"],
                                          ref["ts"], m_rows=np.array([12, 3]), n_rows=cols, threads=threads).y,
                              y4[np.ix_([12, 3], cols)])


def test_gemm_reference_magnitude_sums():
    """The accumulation allowance's S = sum_k |a_k| |b_k|, which the
    comparators get from the oracle on sign-cleared operands, equals the
    binary64 product of the absolute dequantised operands (numpy), for both
    GEMMs and the straight-through gradients; the W4A16 input-rounding term
    uses each weight row's sum of |w|."""
    from nvfp4_testutil import oracle_qat, oracle_w4a16, oracle_w4a4
    w = synth.weight_normal(40, 256, seed=41, outlier_frac=0.02)
    ref = oracle.quantize_fos(w)
    x = synth.act_student_t(9, 256, seed=42)
    a = oracle.quantize_act(x)

    def deq(codes, scales, ts):
        vals = np.array([oracle.e2m1_value(c) for c in range(16)])
        q = np.stack([codes & 15, codes >> 4], axis=-1).reshape(codes.shape[0], -1)
        sv = np.array([oracle.e4m3_value(b) for b in range(256)])[scales]
        return vals[q] * np.repeat(sv, 16, axis=1) * ts
    wd = deq(ref["codes"], ref["scales"], ref["ts"])
    ad = deq(a["codes"], a["scales"], a["ts"])
    xd = oracle.bf16_to_f32(x).astype(np.float64)
    r16 = oracle_w4a16(x, ref["codes"], ref["scales"], ref["ts"])
    assert np.allclose(r16.s, np.abs(xd) @ np.abs(wd).T, rtol=1e-12, atol=0)
    assert np.allclose(r16.y, xd @ wd.T, rtol=1e-9, atol=1e-12)
    assert r16.k == 256
    assert np.allclose(r16.xin, 2.0 ** -39 * np.max(np.abs(xd), axis=1, keepdims=True) * np.abs(wd).sum(axis=1),
                       rtol=1e-12, atol=0)
    r4 = oracle_w4a4(a["codes"], a["scales"], a["ts"], ref["codes"], ref["scales"], ref["ts"])
    assert np.allclose(r4.s, np.abs(ad) @ np.abs(wd).T, rtol=1e-12, atol=0) and r4.k == 256 and r4.xin is None
    rng = np.random.default_rng(43)
    dy = synth.f32_to_bf16_bits(rng.standard_normal((9, 40)).astype(np.float32))
    w_hat = oracle.dequant_bf16(ref["codes"], ref["scales"], ref["ts"])
    x_hat = oracle.dequant_bf16(a["codes"], a["scales"], a["ts"])
    gx, gw = oracle_qat(dy, w_hat, x_hat)
    dyd = oracle.bf16_to_f32(dy).astype(np.float64)
    whd, xhd = oracle.bf16_to_f32(w_hat).astype(np.float64), oracle.bf16_to_f32(x_hat).astype(np.float64)
    assert np.allclose(gx.s, np.abs(dyd) @ np.abs(whd), rtol=1e-12, atol=0) and gx.k == 40
    assert np.allclose(gw.s, np.abs(dyd).T @ np.abs(xhd), rtol=1e-12, atol=0) and gw.k == 9


def test_gemm_tolerance_checker():
    """The comparator every GEMM parity test uses (R14): binary32 outputs
    within 1e-3 of max|ref_row| per row, within 1e-3 (|ref| + rms(ref_row))
    elementwise and within the accumulation allowance
    (ceil(k/16) + 8) 2^-23 S; bf16 outputs one of the two bf16 values that
    bracket ref widened by that allowance; non-finite outputs fail."""
    from nvfp4_testutil import GemmRef, assert_gemm_close, bf16_bracket
    # the bf16 bracket, by hand
    lo, hi = bf16_bracket(np.array([1.0, 1.0 + 2.0 ** -9, -3.1, 0.0, 2.0 ** -130 + 2.0 ** -140, 255.5]))
    assert list(lo) == [1.0, 1.0, -3.109375, 0.0, 2.0 ** -130, 255.0]  # spacing 2^-6 in [2, 4)
    assert list(hi) == [1.0, 1.0 + 2.0 ** -7, -3.09375, 0.0, 2.0 ** -130 + 2.0 ** -133, 256.0]
    # the allowance, by hand
    ref = np.array([[1.0, -0.5, 0.25], [1e-6, -2e-6, 3e-6]])
    g = GemmRef(ref, np.ones_like(ref), 4096)
    assert np.all(g.allowance() == 264 * 2.0 ** -23 + 16 * 2.0 ** -149)
    # binary32: the allowance binds when S is small...
    small = GemmRef(ref, np.abs(ref) * 10, 64)  # acc = 12 * 2^-23 * 10 |ref|, far inside the R14 bounds
    acc = small.allowance()
    assert_gemm_close(ref + 0.99 * acc, small, bf16=False)
    bump = np.zeros_like(ref)
    bump[1, 2] = 1.01
    with pytest.raises(AssertionError):
        assert_gemm_close(ref + bump * acc, small, bf16=False)
    # ...and the R14 clauses bind when S is large
    big = GemmRef(ref, np.full_like(ref, 1e6), 64)
    rms = np.sqrt(np.mean(ref * ref, axis=1, keepdims=True))
    elem = 1e-3 * (np.abs(ref) + rms)
    rowb = 1e-3 * np.max(np.abs(ref), axis=1, keepdims=True)
    tight = np.minimum(elem, rowb)
    assert_gemm_close(ref + 0.99 * tight, big, bf16=False)
    with pytest.raises(AssertionError):  # elementwise clause on a small element of the first row
        assert_gemm_close(ref + np.array([[0, 0, 1.01], [0, 0, 0]]) * elem, big, bf16=False)
    with pytest.raises(AssertionError):  # row clause on the small-scale row
        assert_gemm_close(ref + np.array([[0, 0, 0], [0, 1.01, 0]]) * rowb, big, bf16=False)
    bad = ref.copy()
    bad[0, 1] = np.nan
    with pytest.raises(AssertionError):
        assert_gemm_close(bad, big, bf16=False)
    with pytest.raises(AssertionError):
        assert_gemm_close(ref[:, :2], big, bf16=False)
    with pytest.raises(AssertionError):  # a bare array carries no allowance
        assert_gemm_close(ref, ref, bf16=False)
    # bf16: both neighbours of an exact value pass, the next ones fail
    rng = np.random.default_rng(33)
    exact = rng.standard_normal((6, 50)) * np.exp(rng.uniform(-20, 20, (6, 1)))
    exact_ref = GemmRef(exact, np.abs(exact) * 1e-3, 16)  # allowance far below half a bf16 step
    lo, hi = bf16_bracket(exact)
    assert_gemm_close(lo, exact_ref, bf16=True)
    assert_gemm_close(hi, exact_ref, bf16=True)
    rounded = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(exact.astype(np.float32))).astype(np.float64)
    assert_gemm_close(rounded, exact_ref, bf16=True)
    below, _ = bf16_bracket(np.nextafter(lo, -np.inf))
    with pytest.raises(AssertionError):
        assert_gemm_close(np.where(np.arange(50) == 7, below, lo), exact_ref, bf16=True)
    # a near-zero element: the allowance lets the accumulated value round either way
    z = np.array([[2.0 ** -40, 1.0]])
    zr = GemmRef(z, np.array([[1.0, 1.0]]), 16)  # allowance ~ 2^-20 >> 2^-40
    assert_gemm_close(np.array([[-2.0 ** -22, 1.0]]), zr, bf16=True)
    with pytest.raises(AssertionError):
        assert_gemm_close(np.array([[-2.0 ** -15, 1.0]]), zr, bf16=True)


def test_silu_mul_tolerance_checker():
    """The gated projection's comparator: |y - silu(g) u| within
    1.1 eg (|u| + eu) + |silu(g)| eu + 2^-19 (1 + |g|) |silu(g) u| (eg, eu the
    GEMM allowances), bf16 in the bracket of that interval; gate and up
    swapped fail."""
    from nvfp4_testutil import GemmRef, assert_silu_mul_close, bf16_bracket, silu_mul_allowance, silu_mul_ref
    rng = np.random.default_rng(34)
    gy = rng.standard_normal((3, 40)) * 3
    uy = rng.standard_normal((3, 40))
    g = GemmRef(gy, np.abs(gy) * 4, 256)
    u = GemmRef(uy, np.abs(uy) * 4, 256)
    y = silu_mul_ref(gy, uy)
    allow = silu_mul_allowance(g, u)
    eg, eu = g.allowance(), u.allowance()
    sg = silu_mul_ref(gy, np.ones_like(gy))
    assert np.allclose(allow, 1.1 * eg * (np.abs(uy) + eu) + np.abs(sg) * eu +
                       2.0 ** -19 * (1 + np.abs(gy)) * np.abs(y) + 2.0 ** -140, rtol=1e-15, atol=0)
    assert_silu_mul_close(y + 0.99 * allow, g, u, bf16=False)
    bump = np.zeros_like(y)
    bump[2, 7] = 1.01
    with pytest.raises(AssertionError):
        assert_silu_mul_close(y + bump * allow, g, u, bf16=False)
    with pytest.raises(AssertionError):
        assert_silu_mul_close(silu_mul_ref(uy, gy), g, u, bf16=False)  # gate and up swapped
    lo, hi = bf16_bracket(y)
    assert_silu_mul_close(lo, g, u, bf16=True)
    assert_silu_mul_close(hi, g, u, bf16=True)

