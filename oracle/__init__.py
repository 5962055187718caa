"""CPU oracle for the NVFP4 linear-layer path -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline may import this package.  The product library never loads it, and it
shares no code with the CUDA path.  The arithmetic lives in
``nvfp4_oracle.c`` (plain C, binary32 for the quantiser's decisions, binary64
for the GEMM references); this module compiles it with gcc and wraps it with
ctypes + numpy.

Method sources (web pages about the SOAR 2026 inference contest):
  * "SOAR 2026 Recap ...", section "1. Quantization and GEMM dispatch", and
    section "3. EAGLE-3 speculative decoding ..." (NVFP4 QAT, for the
    dequantisation and straight-through gradients);
  * "SOAR Weekly Champion Notes 07 ... NVFP4 Quantization Improvements",
    sections "01 Background", "02 FourOverSix" and "03 How we integrated it"
    (GPTQ inside the FourOverSix scales).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

DEFAULT_DIVISOR = 6.0 * 448.0

# gcc flags: no fused multiply-add contraction and no fast-math, so every
# binary32 step rounds exactly once as written.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-fexcess-precision=standard", "-Wall"]


def build(force: bool = False) -> str:
    """Compile liboracle.so next to the source (gcc only)."""
    with _lock:
        if force or not os.path.exists(_LIB_PATH) or \
                os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        u8p = ctypes.POINTER(ctypes.c_uint8)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f32p = ctypes.POINTER(ctypes.c_float)
        f64p = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_value.restype = ctypes.c_float
        lib.oracle_e2m1_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e2m1_value.restype = ctypes.c_double
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_value.restype = ctypes.c_double
        lib.oracle_e2m1_encode.argtypes = [ctypes.c_float]
        lib.oracle_e2m1_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_block_sse.argtypes = [f32p, ctypes.c_uint8, ctypes.c_float, u8p]
        lib.oracle_block_sse.restype = ctypes.c_float
        lib.oracle_block_scale_m6.argtypes = [f32p, ctypes.c_float]
        lib.oracle_block_scale_m6.restype = ctypes.c_uint8
        lib.oracle_fos_block.argtypes = [f32p, ctypes.c_float, u8p, u8p, u8p, u8p, u8p, f32p, f32p]
        lib.oracle_fos_block.restype = None
        lib.oracle_tensor_scale.argtypes = [u16p, i64, ctypes.c_float, f32p]
        lib.oracle_tensor_scale.restype = ctypes.c_int
        lib.oracle_quantize_fos.argtypes = [u16p, i64, i64, ctypes.c_float, u8p, u8p, u8p, f32p,
                                            ctypes.POINTER(ctypes.c_uint64)]
        lib.oracle_quantize_fos.restype = ctypes.c_int
        lib.oracle_quantize_rows.argtypes = [u16p, i64, i64, ctypes.c_float, ctypes.c_int, u8p, u8p, u8p]
        lib.oracle_quantize_rows.restype = ctypes.c_uint64
        lib.oracle_quantize_act.argtypes = [u16p, i64, i64, ctypes.c_float, u8p, u8p, f32p]
        lib.oracle_quantize_act.restype = ctypes.c_int
        lib.oracle_scales_mma_bytes.argtypes = [i64, i64]
        lib.oracle_scales_mma_bytes.restype = i64
        lib.oracle_scales_to_mma.argtypes = [u8p, i64, i64, u8p]
        lib.oracle_scales_to_mma.restype = None
        lib.oracle_gemm_w4a16.argtypes = [u16p, i64, i64, u8p, u8p, ctypes.c_float, i64, f64p]
        lib.oracle_gemm_w4a16.restype = ctypes.c_int
        lib.oracle_gemm_w4a16_rows.argtypes = [u16p, ctypes.POINTER(ctypes.c_int64), i64, i64, u8p,
                                               u8p, ctypes.c_float, i64, f64p]
        lib.oracle_gemm_w4a16_rows.restype = ctypes.c_int
        lib.oracle_gemm_w4a4.argtypes = [u8p, u8p, ctypes.c_float, i64, u8p, u8p, ctypes.c_float,
                                         i64, i64, f64p]
        lib.oracle_gemm_w4a4.restype = ctypes.c_int
        lib.oracle_dequant_bf16.argtypes = [u8p, u8p, ctypes.c_float, i64, i64, u16p]
        lib.oracle_dequant_bf16.restype = ctypes.c_int
        lib.oracle_gptq_fos.argtypes = [u16p, i64, i64, f32p, ctypes.c_float, i64, u8p, u8p, f32p, f32p]
        lib.oracle_gptq_fos_ref64.argtypes = [u16p, i64, i64, f32p, ctypes.c_double, u8p, ctypes.c_float, u8p,
                                              ctypes.c_double, u8p, u8p]
        lib.oracle_gptq_fos.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


class OracleError(RuntimeError):
    def __init__(self, status: int):
        super().__init__(f"oracle status {status}")
        self.status = status


# ---------------------------------------------------------------- formats ---

def bf16_value(bits: int) -> float:
    return _load().oracle_bf16_value(bits)


def e2m1_value(code: int) -> float:
    return _load().oracle_e2m1_value(code)


def e4m3_value(byte: int) -> float:
    return _load().oracle_e4m3_value(byte)


def e2m1_encode(v: float) -> int:
    return _load().oracle_e2m1_encode(v)


def e4m3_encode(v: float) -> int:
    return _load().oracle_e4m3_encode(v)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact: bf16 is the top half of binary32)."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------ blocks ---

def block_sse(x, scale_byte: int, ts: float):
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.shape == (16,)
    q = np.zeros(16, np.uint8)
    sse = _load().oracle_block_sse(_ptr(x, ctypes.c_float), scale_byte, ts, _ptr(q, ctypes.c_uint8))
    return float(sse), q


def fos_block(x, ts: float) -> dict:
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.shape == (16,)
    q = np.zeros(16, np.uint8)
    s = ctypes.c_uint8()
    c = ctypes.c_uint8()
    s6 = ctypes.c_uint8()
    s4 = ctypes.c_uint8()
    e6 = ctypes.c_float()
    e4 = ctypes.c_float()
    _load().oracle_fos_block(_ptr(x, ctypes.c_float), ts, _ptr(q, ctypes.c_uint8), ctypes.byref(s),
                             ctypes.byref(c), ctypes.byref(s6), ctypes.byref(s4), ctypes.byref(e6),
                             ctypes.byref(e4))
    return dict(codes=q, scale=s.value, choice=c.value, s6=s6.value, s4=s4.value,
                sse6=e6.value, sse4=e4.value)


# ----------------------------------------------------------------- tensors ---

def tensor_scale(x_bits: np.ndarray, divisor: float = DEFAULT_DIVISOR) -> float:
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    ts = ctypes.c_float()
    st = _load().oracle_tensor_scale(_ptr(x_bits, ctypes.c_uint16), x_bits.size, divisor,
                                     ctypes.byref(ts))
    if st:
        raise OracleError(st)
    return ts.value


def quantize_fos(w_bits: np.ndarray, divisor: float = DEFAULT_DIVISOR) -> dict:
    """FourOverSix NVFP4 quantisation of a bf16 [N, K] weight given as uint16 bits."""
    w_bits = np.ascontiguousarray(w_bits, dtype=np.uint16)
    N, K = w_bits.shape
    codes = np.zeros((N, K // 2), np.uint8)
    scales = np.zeros((N, K // 16), np.uint8)
    choice = np.zeros((N, K // 16), np.uint8)
    ts = ctypes.c_float()
    m4 = ctypes.c_uint64()
    st = _load().oracle_quantize_fos(_ptr(w_bits, ctypes.c_uint16), N, K, divisor,
                                     _ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_uint8),
                                     _ptr(choice, ctypes.c_uint8), ctypes.byref(ts),
                                     ctypes.byref(m4))
    if st:
        raise OracleError(st)
    return dict(codes=codes, scales=scales, choice=choice, ts=ts.value, m4_count=m4.value)


def quantize_rows(x_bits: np.ndarray, ts: float, fos: bool, threads: int = 1) -> dict:
    """Quantise every row of a bf16 matrix with a given tensor scale (FourOverSix
    when `fos`, else M=6 only).  Rows are independent, so they may be split
    across threads (the C call releases the GIL); the result does not depend on
    the split."""
    import concurrent.futures as cf
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    R, K = x_bits.shape
    codes = np.zeros((R, K // 2), np.uint8)
    scales = np.zeros((R, K // 16), np.uint8)
    choice = np.zeros((R, K // 16), np.uint8)
    lib = _load()
    bounds = np.linspace(0, R, max(1, min(threads, R)) + 1).astype(np.int64)

    def run(i):
        a, b = int(bounds[i]), int(bounds[i + 1])
        if a == b:
            return 0
        return lib.oracle_quantize_rows(_ptr(x_bits[a:b], ctypes.c_uint16), b - a, K, ts, int(fos),
                                        _ptr(codes[a:b], ctypes.c_uint8), _ptr(scales[a:b], ctypes.c_uint8),
                                        _ptr(choice[a:b], ctypes.c_uint8))
    with cf.ThreadPoolExecutor(max_workers=len(bounds) - 1) as ex:
        m4 = sum(ex.map(run, range(len(bounds) - 1)))
    return dict(codes=codes, scales=scales, choice=choice, ts=ts, m4_count=int(m4))


def quantize_act(x_bits: np.ndarray, divisor: float = DEFAULT_DIVISOR) -> dict:
    """Standard (M=6) NVFP4 quantisation of bf16 activations [M, K]."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, K = x_bits.shape
    codes = np.zeros((M, K // 2), np.uint8)
    scales = np.zeros((M, K // 16), np.uint8)
    ts = ctypes.c_float()
    st = _load().oracle_quantize_act(_ptr(x_bits, ctypes.c_uint16), M, K, divisor,
                                     _ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_uint8),
                                     ctypes.byref(ts))
    if st:
        raise OracleError(st)
    return dict(codes=codes, scales=scales, ts=ts.value)


def scales_to_mma(scales: np.ndarray, K: int) -> np.ndarray:
    """Logical [R, K/16] scales -> the 128x4-tiled tensor-core layout (flat bytes)."""
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    R = scales.shape[0]
    lib = _load()
    out = np.zeros(lib.oracle_scales_mma_bytes(R, K), np.uint8)
    lib.oracle_scales_to_mma(_ptr(scales, ctypes.c_uint8), R, K, _ptr(out, ctypes.c_uint8))
    return out


def gemm_w4a16(x_bits: np.ndarray, codes: np.ndarray, scales: np.ndarray, ts: float) -> np.ndarray:
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, K = x_bits.shape
    N = codes.shape[0]
    y = np.zeros((M, N), np.float64)
    st = _load().oracle_gemm_w4a16(_ptr(x_bits, ctypes.c_uint16), M, K,
                                   _ptr(np.ascontiguousarray(codes), ctypes.c_uint8),
                                   _ptr(np.ascontiguousarray(scales), ctypes.c_uint8), ts, N,
                                   _ptr(y, ctypes.c_double))
    if st:
        raise OracleError(st)
    return y


def gemm_w4a16_rows(x_bits: np.ndarray, rows, codes: np.ndarray, scales: np.ndarray,
                    ts: float) -> np.ndarray:
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    K = x_bits.shape[1]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    N = codes.shape[0]
    y = np.zeros((rows.size, N), np.float64)
    st = _load().oracle_gemm_w4a16_rows(_ptr(x_bits, ctypes.c_uint16), _ptr(rows, ctypes.c_int64),
                                        rows.size, K,
                                        _ptr(np.ascontiguousarray(codes), ctypes.c_uint8),
                                        _ptr(np.ascontiguousarray(scales), ctypes.c_uint8), ts, N,
                                        _ptr(y, ctypes.c_double))
    if st:
        raise OracleError(st)
    return y


def gemm_w4a4(a_codes, a_scales, a_ts, w_codes, w_scales, w_ts) -> np.ndarray:
    a_codes = np.ascontiguousarray(a_codes, dtype=np.uint8)
    M = a_codes.shape[0]
    K = a_codes.shape[1] * 2
    N = w_codes.shape[0]
    y = np.zeros((M, N), np.float64)
    st = _load().oracle_gemm_w4a4(_ptr(a_codes, ctypes.c_uint8),
                                  _ptr(np.ascontiguousarray(a_scales, dtype=np.uint8), ctypes.c_uint8),
                                  a_ts, M,
                                  _ptr(np.ascontiguousarray(w_codes, dtype=np.uint8), ctypes.c_uint8),
                                  _ptr(np.ascontiguousarray(w_scales, dtype=np.uint8), ctypes.c_uint8),
                                  w_ts, N, K, _ptr(y, ctypes.c_double))
    if st:
        raise OracleError(st)
    return y


def dequant_bf16(codes: np.ndarray, scales: np.ndarray, ts: float) -> np.ndarray:
    """NVFP4 [R, K] (codes [R, K/2], logical scales [R, K/16]) -> bf16 bits,
    value(code) * value(scale) exact, times ts rounded to binary32, then to
    bfloat16 (the operand of the QAT backward's bf16 GEMMs)."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    R, K = codes.shape[0], codes.shape[1] * 2
    out = np.zeros((R, K), np.uint16)
    st = _load().oracle_dequant_bf16(_ptr(codes, ctypes.c_uint8),
                                     _ptr(np.ascontiguousarray(scales, dtype=np.uint8), ctypes.c_uint8), ts,
                                     R, K, _ptr(out, ctypes.c_uint16))
    if st:
        raise OracleError(st)
    return out


def qat_backward(dy_bits: np.ndarray, w_hat_bits: np.ndarray, x_hat_bits: np.ndarray):
    """Gradients of Y = X_hat W_hat^T under the straight-through estimator
    ("SOAR 2026 Recap ...", section "3. EAGLE-3 speculative decoding and
    hybrid architecture adaptation", paragraph "NVFP4 QAT": the FP4 forward's
    gradients pass straight through to the bf16 master weights): dX = dY W_hat and
    dW = dY^T X_hat, binary64 products (numpy matmul) of the bf16 operands.
    dy [M, N], w_hat [N, K], x_hat [M, K] as bf16 bits."""
    dy = bf16_to_f32(dy_bits).astype(np.float64)
    w = bf16_to_f32(w_hat_bits).astype(np.float64)
    x = bf16_to_f32(x_hat_bits).astype(np.float64)
    return dy @ w, dy.T @ x


def gptq_fos(w_bits: np.ndarray, H: np.ndarray, damp: float = 0.01, block: int = 128,
             want_u: bool = False) -> dict:
    """GPTQ inside FourOverSix scales ("SOAR Weekly Champion Notes 07 ...",
    section "03 How we integrated it": each block's M is fixed first, then
    GPTQ runs within it).  w_bits bf16 [N, K]; H float32 [K, K] (the layer's
    Hessian, e.g. 2 X^T X / T from calibration activations).  Returns codes,
    logical scales, ts (and U, the upper Cholesky factor of the damped
    inverse Hessian) computed in the binary32 order stated in nvfp4_oracle.c."""
    w_bits = np.ascontiguousarray(w_bits, dtype=np.uint16)
    N, K = w_bits.shape
    H = np.ascontiguousarray(H, dtype=np.float32)
    assert H.shape == (K, K)
    codes = np.zeros((N, K // 2), np.uint8)
    scales = np.zeros((N, K // 16), np.uint8)
    ts = np.zeros(1, np.float32)
    U = np.zeros((K, K), np.float32) if want_u else None
    st = _load().oracle_gptq_fos(_ptr(w_bits, ctypes.c_uint16), N, K, _ptr(H, ctypes.c_float), damp, block,
                                 _ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_uint8),
                                 _ptr(ts, ctypes.c_float),
                                 _ptr(U, ctypes.c_float) if want_u else None)
    if st:
        raise OracleError(st)
    out = {"codes": codes, "scales": scales, "ts": float(ts[0])}
    if want_u:
        out["U"] = U
    return out


def gptq_fos_ref64(w_bits: np.ndarray, H: np.ndarray, scales: np.ndarray, ts: float, damp: float = 0.01,
                   follow: np.ndarray | None = None, delta: float = 1e-3) -> dict:
    """The same GPTQ written plainly in binary64, unblocked (nvfp4_oracle.c,
    oracle_gptq_fos_ref64), on given FourOverSix scales and tensor scale.
    With `follow` (another run's codes), elements whose quotient lies within
    `delta` of an E2M1 rounding midpoint take the followed code and are
    flagged in "near"; a followed code that is not one of the two values
    either side of that midpoint raises."""
    w_bits = np.ascontiguousarray(w_bits, dtype=np.uint16)
    N, K = w_bits.shape
    H = np.ascontiguousarray(H, dtype=np.float32)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    assert H.shape == (K, K) and scales.shape == (N, K // 16)
    codes = np.zeros((N, K // 2), np.uint8)
    near = np.zeros((N, K), np.uint8)
    fol = None if follow is None else np.ascontiguousarray(follow, dtype=np.uint8)
    st = _load().oracle_gptq_fos_ref64(_ptr(w_bits, ctypes.c_uint16), N, K, _ptr(H, ctypes.c_float), damp,
                                       _ptr(scales, ctypes.c_uint8), ts,
                                       None if fol is None else _ptr(fol, ctypes.c_uint8), delta,
                                       _ptr(codes, ctypes.c_uint8), _ptr(near, ctypes.c_uint8))
    if st:
        raise OracleError(st)
    return {"codes": codes, "near": near.astype(bool)}
