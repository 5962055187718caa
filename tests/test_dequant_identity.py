"""The arithmetic identity behind the GPU dequantiser's value formation.

The bf16 dequantisation (nvfp4_dequantize and the QAT backward's operands)
forms value(code) * value(scale) without an integer-to-float conversion: the
E2M1 code's magnitude bits placed at binary32 bits 24:22 and its sign at bit
31 read as value(code) * 2^-126 exactly (0.5 lands in the subnormal range),
the product with the E4M3 scale is exact, and times 2^126 restores
value(code) * value(scale).  This checks, in binary32 with subnormals, that
the three steps give the same bits as the direct product for every code and
every finite E4M3 scale, and that the final multiply by a tensor scale then
rounds identically.  The E2M1 value set is the one "SOAR Weekly Champion Notes
07", section "01 Background", prints; the E4M3 values follow the format
definition (bias 7, subnormals m * 2^-9)."""
import numpy as np

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def e4m3_value(b):
    e, m = (b >> 3) & 15, b & 7
    return m * 2.0 ** -9 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)


def placed(code):
    bits = np.uint32(((code & 7) << 22) | ((code & 8) << 28))
    return bits.view(np.float32)


def direct(code, s):
    mag = np.float32(E2M1[code & 7])
    return (-mag if code & 8 else mag) * s


def test_bit_placement_reads_value_times_2_pow_minus_126():
    for code in range(16):
        v = placed(code)
        want = (-1.0 if code & 8 else 1.0) * E2M1[code & 7] * 2.0 ** -126
        assert float(v) == want
        assert np.signbit(v) == bool(code & 8)  # code 8 is -0


def test_placed_product_equals_direct_product_bitwise():
    two126 = np.float32(2.0 ** 126)
    with np.errstate(all="raise"):
        for code in range(16):
            v = placed(code)
            for sb in range(0x7F):  # every finite non-negative E4M3 byte
                s = np.float32(e4m3_value(sb))
                p = np.float32(v * s)
                assert float(p) == float(v) * float(s)  # exact, subnormal or not
                q = np.float32(p * two126)
                d = direct(code, s)
                assert q.view(np.uint32) == d.view(np.uint32), (code, sb)


def test_tensor_scale_step_rounds_identically():
    rng = np.random.default_rng(5)
    two126 = np.float32(2.0 ** 126)
    ts_values = np.concatenate([rng.uniform(1e-6, 1e-1, 64), [2.0 ** -126, 1.0, 3.0e3]]).astype(np.float32)
    for ts in ts_values:
        for code in (1, 7, 9, 15):
            for sb in (1, 8, 0x38, 0x7E):
                s = np.float32(e4m3_value(sb))
                a = np.float32(np.float32(np.float32(placed(code) * s) * two126) * ts)
                b = np.float32(direct(code, s) * ts)
                assert a.view(np.uint32) == b.view(np.uint32)
