"""Helpers shared by the GPU parity tests: device transfers, oracle
references computed in parallel threads, and the GEMM tolerance check."""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np

import oracle

THREADS = max(1, min(32, os.cpu_count() or 1))

# GEMM bar (R14 of the design notes), against the binary64 product of the
# exactly dequantised operands:
#   binary32 outputs: per output row max |y - ref| <= 1e-3 * max |ref_row|, and
#     elementwise |y - ref| <= 1e-3 * |ref| + 1e-3 * rms(ref_row), and
#     elementwise |y - ref| <= the accumulation allowance below;
#   bf16 outputs: y is one of the two bf16 values that bracket ref, widened
#     by the accumulation allowance ("compared after rounding").
# Accumulation allowance, derived from the contraction length k: the kernels
# add their exact products into binary32 accumulators one MMA step of at most
# 16 products at a time, and every partial sum and addend is bounded by
# S = sum_k |a_k| |b_k|; allowing each step one rounding of relative size
# 2^-23 (truncating hardware accumulation included) and up to 8 further
# roundings (split-K partial sums, the tensor scales, a power-of-two rescale)
# gives |y32 - ref| <= (ceil(k / 16) + 8) * 2^-23 * S, plus 16 * 2^-149 for
# results in the binary32 subnormal range and, where a kernel rounds tiny
# activations to f16 subnormals, 2^-39 * max|x_row| * sum_k |w_k|.
GEMM_REL_TOL = 1e-3


class GemmRef:
    """A GEMM's binary64 reference `y` with what its allowance needs: `s`, the
    binary64 sum of |a_k| |b_k| per output; `k`, the contraction length; `xin`
    (optional), the bound on input rounding inside the kernel."""

    def __init__(self, y, s, k, xin=None):
        self.y, self.s, self.k, self.xin = y, s, k, xin

    def rows(self, idx):
        return GemmRef(self.y[idx], self.s[idx], self.k, None if self.xin is None else self.xin[idx])

    def cols(self, idx):
        return GemmRef(self.y[:, idx], self.s[:, idx], self.k, None if self.xin is None else self.xin[:, idx])

    def allowance(self):
        a = (np.ceil(self.k / 16) + 8) * 2.0 ** -23 * self.s + 16 * 2.0 ** -149
        return a if self.xin is None else a + self.xin


def to_dev(bits: np.ndarray):
    """uint16 bf16 bits (numpy) -> contiguous CUDA bfloat16 tensor."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.cuda()


def to_np_u8(t) -> np.ndarray:
    return t.detach().cpu().numpy().astype(np.uint8)


def y_to_np(y) -> np.ndarray:
    import torch
    return y.detach().float().cpu().numpy().astype(np.float64) if y.dtype != torch.float32 \
        else y.detach().cpu().numpy().astype(np.float64)


def _by_rows(M, threads, run_rows, n_out):
    bounds = np.linspace(0, M, max(1, min(threads, M)) + 1).astype(int)

    def run(i):
        a, b = bounds[i], bounds[i + 1]
        return np.zeros((0, n_out)) if a == b else run_rows(a, b)
    with cf.ThreadPoolExecutor(len(bounds) - 1) as ex:
        return np.concatenate(list(ex.map(run, range(len(bounds) - 1))), axis=0)


def _mag_codes(codes):
    """E2M1 codes with both nibbles' sign bits cleared: the magnitudes."""
    return np.ascontiguousarray(codes & np.uint8(0x77))


def _mag_bits(bits):
    """bf16 bit patterns with the sign bit cleared."""
    return np.ascontiguousarray(bits & np.uint16(0x7FFF))


def oracle_w4a16(x_bits, codes, scales, ts, n_rows=None, threads=THREADS):
    """binary64 reference of X @ dequant(W)^T with its accumulation allowance
    (a GemmRef); optionally only for the weight rows `n_rows` (output
    columns), split over threads by activation row.  The W4A16 kernels round
    tiny activations to f16 subnormals, so xin bounds that too."""
    if n_rows is not None:
        codes, scales = codes[n_rows], scales[n_rows]
    codes = np.ascontiguousarray(codes)
    scales = np.ascontiguousarray(scales)
    x_bits = np.ascontiguousarray(x_bits)
    M, K, N = x_bits.shape[0], x_bits.shape[1], codes.shape[0]
    y = _by_rows(M, threads, lambda a, b: oracle.gemm_w4a16(x_bits[a:b], codes, scales, ts), N)
    xm, cm = _mag_bits(x_bits), _mag_codes(codes)
    s = _by_rows(M, threads, lambda a, b: oracle.gemm_w4a16(xm[a:b], cm, scales, ts), N)
    wsum = oracle.gemm_w4a16(np.full((1, K), 0x3F80, np.uint16), cm, scales, ts)  # sum_k |w_nk|
    xmax = np.max(np.abs(oracle.bf16_to_f32(x_bits).astype(np.float64)), axis=1, keepdims=True) if M else \
        np.zeros((0, 1))
    return GemmRef(y, s, K, 2.0 ** -39 * xmax * wsum)


def oracle_w4a4(a_codes, a_scales, a_ts, w_codes, w_scales, w_ts, m_rows=None, n_rows=None, threads=THREADS):
    """binary64 reference of dequant(A) @ dequant(W)^T with its accumulation
    allowance (a GemmRef); optionally only rows `m_rows` / columns `n_rows`."""
    if m_rows is not None:
        a_codes, a_scales = a_codes[m_rows], a_scales[m_rows]
    if n_rows is not None:
        w_codes, w_scales = w_codes[n_rows], w_scales[n_rows]
    a_codes, a_scales = np.ascontiguousarray(a_codes), np.ascontiguousarray(a_scales)
    w_codes, w_scales = np.ascontiguousarray(w_codes), np.ascontiguousarray(w_scales)
    M, N, K = a_codes.shape[0], w_codes.shape[0], 2 * a_codes.shape[1]
    y = _by_rows(M, threads, lambda a, b: oracle.gemm_w4a4(a_codes[a:b], a_scales[a:b], a_ts, w_codes, w_scales,
                                                           w_ts), N)
    am, wm = _mag_codes(a_codes), _mag_codes(w_codes)
    s = _by_rows(M, threads, lambda a, b: oracle.gemm_w4a4(am[a:b], a_scales[a:b], a_ts, wm, w_scales, w_ts), N)
    return GemmRef(y, s, K)


def oracle_qat(dy_bits, w_hat_bits, x_hat_bits):
    """The straight-through gradients dX = dY W_hat and dW = dY^T X_hat as
    GemmRefs (contraction over N and over M)."""
    dx, dw = oracle.qat_backward(dy_bits, w_hat_bits, x_hat_bits)
    sx, sw = oracle.qat_backward(_mag_bits(dy_bits), _mag_bits(w_hat_bits), _mag_bits(x_hat_bits))
    M, N = dy_bits.shape
    return GemmRef(dx, sx, N), GemmRef(dw, sw, M)


def bf16_bracket(v: np.ndarray):
    """(largest bf16 value <= v, smallest bf16 value >= v) as binary64, for
    finite v within the bf16 range: 8 significant bits, spacing fixed at
    2^-133 below 2^-126."""
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.where(a > 0, np.maximum(e, -126.0), -126.0)
    q = 2.0 ** (e - 7)
    return np.floor(v / q) * q, np.ceil(v / q) * q


def gemm_errors(y: np.ndarray, ref: GemmRef, bf16: bool):
    """Returns (worst normwise row error, mask of failing elements)."""
    r = ref.y
    err = np.abs(y - r)
    acc = ref.allowance()
    scale = np.max(np.abs(r), axis=1, keepdims=True) if r.size else np.zeros((r.shape[0], 1))
    if bf16:
        lo, _ = bf16_bracket(r - acc)
        _, hi = bf16_bracket(r + acc)
        bad = (y < lo) | (y > hi)
        excess = np.maximum(err - np.maximum(hi - r, r - lo), 0)
    else:
        rms = np.sqrt(np.mean(r * r, axis=1, keepdims=True)) if r.size else np.zeros((r.shape[0], 1))
        bad = (err > GEMM_REL_TOL * scale) | (err > GEMM_REL_TOL * (np.abs(r) + rms)) | (err > acc)
        excess = err
    with np.errstate(divide="ignore", invalid="ignore"):
        rel = np.where(scale > 0, np.max(excess, axis=1, keepdims=True) / scale, 0.0) if r.size else np.zeros(1)
    return float(np.max(rel)) if rel.size else 0.0, bad


def assert_gemm_close(y: np.ndarray, ref: GemmRef, bf16: bool, what: str = ""):
    assert isinstance(ref, GemmRef), "the comparator needs the reference's accumulation allowance"
    assert y.shape == ref.y.shape, (y.shape, ref.y.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    worst, bad = gemm_errors(y, ref, bf16)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        acc = ref.allowance()
        detail = ", ".join(f"[{i},{j}] y={y[i, j]!r} ref={ref.y[i, j]!r} acc={acc[i, j]:.3g}" for i, j in idx)
        raise AssertionError(f"{what}: {int(bad.sum())} elements outside tolerance "
                             f"(worst normwise rel {worst:.3g}); e.g. {detail}")
    return worst


# silu(G) * U for G, U from a GEMM with allowances eg, eu (above): as
# silu'(g) lies in [-0.1, 1.1] and |silu(g)| <= |g|,
#   |silu(g') u' - silu(g) u| <= 1.1 eg (|u| + eu) + |silu(g)| eu,
# and the binary32 evaluation (fast exponential of -g: relative error about
# |g| 2^-24 + 2^-22; fast division 2^-21; the product 2^-24) adds at most
# 2^-19 (1 + |g|) |silu(g) u|.  bf16 outputs must lie in the bf16 bracket of
# that interval.


def silu_mul_ref(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """binary64 silu(g) * u = g / (1 + e^-g) * u."""
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g)) * u


def silu_mul_allowance(g: GemmRef, u: GemmRef) -> np.ndarray:
    eg, eu = g.allowance(), u.allowance()
    sg = silu_mul_ref(g.y, np.ones_like(g.y))
    ref = sg * u.y
    return 1.1 * eg * (np.abs(u.y) + eu) + np.abs(sg) * eu + 2.0 ** -19 * (1 + np.abs(g.y)) * np.abs(ref) + \
        2.0 ** -140


def assert_silu_mul_close(y: np.ndarray, g: GemmRef, u: GemmRef, bf16: bool, what: str = ""):
    """y against silu(g) * u elementwise, g and u the binary64 GEMM references
    of the gate and up halves."""
    assert isinstance(g, GemmRef) and isinstance(u, GemmRef)
    ref = silu_mul_ref(g.y, u.y)
    assert y.shape == ref.shape, (y.shape, ref.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    allow = silu_mul_allowance(g, u)
    if bf16:
        lo, _ = bf16_bracket(ref - allow)
        _, hi = bf16_bracket(ref + allow)
        bad = (y < lo) | (y > hi)
    else:
        bad = np.abs(y - ref) > allow
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = ", ".join(f"[{i},{j}] y={y[i, j]!r} ref={ref[i, j]!r} allow={allow[i, j]:.3g}" for i, j in idx)
        raise AssertionError(f"{what}: {int(bad.sum())} elements outside tolerance; e.g. {detail}")
    scale = np.max(np.abs(ref), axis=1, keepdims=True) if ref.size else np.zeros((ref.shape[0], 1))
    with np.errstate(divide="ignore", invalid="ignore"):
        rel = np.where(scale > 0, np.max(np.abs(y - ref), axis=1, keepdims=True) / scale, 0.0) if ref.size \
            else np.zeros(1)
    return float(np.max(rel)) if rel.size else 0.0
