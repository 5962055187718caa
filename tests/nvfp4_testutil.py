"""Helpers shared by the GPU parity tests: device transfers, oracle
references computed in parallel threads, and the GEMM tolerance check."""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np

import oracle

THREADS = max(1, min(32, os.cpu_count() or 1))

# GEMM bar: outputs within a normwise relative error of 1e-3 of the binary64
# oracle (per output row: max |y - ref| <= 1e-3 * max |ref|); bf16 outputs may
# in addition differ by the half-ulp of bf16 rounding of the exact value.
GEMM_REL_TOL = 1e-3


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


def oracle_w4a16(x_bits, codes, scales, ts, n_rows=None, threads=THREADS):
    """binary64 reference of X @ dequant(W)^T; optionally only for the weight
    rows `n_rows` (output columns), split over threads by activation row."""
    if n_rows is not None:
        codes, scales = codes[n_rows], scales[n_rows]
    codes = np.ascontiguousarray(codes)
    scales = np.ascontiguousarray(scales)
    M = x_bits.shape[0]
    bounds = np.linspace(0, M, max(1, min(threads, M)) + 1).astype(int)

    def run(i):
        a, b = bounds[i], bounds[i + 1]
        if a == b:
            return np.zeros((0, codes.shape[0]))
        return oracle.gemm_w4a16(x_bits[a:b], codes, scales, ts)
    with cf.ThreadPoolExecutor(len(bounds) - 1) as ex:
        return np.concatenate(list(ex.map(run, range(len(bounds) - 1))), axis=0)


def oracle_w4a4(a_codes, a_scales, a_ts, w_codes, w_scales, w_ts, m_rows=None, n_rows=None, threads=THREADS):
    if m_rows is not None:
        a_codes, a_scales = a_codes[m_rows], a_scales[m_rows]
    if n_rows is not None:
        w_codes, w_scales = w_codes[n_rows], w_scales[n_rows]
    a_codes, a_scales = np.ascontiguousarray(a_codes), np.ascontiguousarray(a_scales)
    w_codes, w_scales = np.ascontiguousarray(w_codes), np.ascontiguousarray(w_scales)
    M = a_codes.shape[0]
    bounds = np.linspace(0, M, max(1, min(threads, M)) + 1).astype(int)

    def run(i):
        a, b = bounds[i], bounds[i + 1]
        if a == b:
            return np.zeros((0, w_codes.shape[0]))
        return oracle.gemm_w4a4(a_codes[a:b], a_scales[a:b], a_ts, w_codes, w_scales, w_ts)
    with cf.ThreadPoolExecutor(len(bounds) - 1) as ex:
        return np.concatenate(list(ex.map(run, range(len(bounds) - 1))), axis=0)


def bf16_half_ulp(ref: np.ndarray) -> np.ndarray:
    """Half a bf16 ulp at each reference value: 2^(e-8) for binary exponent
    e, and 2^-134 in the subnormal range (below 2^-126 the spacing is fixed at
    2^-133), also at zero."""
    a = np.abs(ref)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.where(a > 0, np.maximum(e, -126.0), -126.0)
    return 2.0 ** (e - 8)


def gemm_errors(y: np.ndarray, ref: np.ndarray, bf16: bool):
    """Returns (worst normwise row error, mask of failing elements)."""
    scale = np.max(np.abs(ref), axis=1, keepdims=True)
    err = np.abs(y - ref)
    allow = GEMM_REL_TOL * scale + (bf16_half_ulp(ref) if bf16 else 0.0)
    bad = err > allow
    with np.errstate(divide="ignore", invalid="ignore"):
        rel = np.where(scale > 0, np.max(np.maximum(err - (bf16_half_ulp(ref) if bf16 else 0.0), 0), axis=1,
                                         keepdims=True) / scale, 0.0)
    return float(np.max(rel)) if rel.size else 0.0, bad


def assert_gemm_close(y: np.ndarray, ref: np.ndarray, bf16: bool, what: str = ""):
    assert y.shape == ref.shape, (y.shape, ref.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    worst, bad = gemm_errors(y, ref, bf16)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = ", ".join(f"[{i},{j}] y={y[i, j]!r} ref={ref[i, j]!r}" for i, j in idx)
        raise AssertionError(f"{what}: {int(bad.sum())} elements outside tolerance "
                             f"(worst normwise rel {worst:.3g}); e.g. {detail}")
    return worst


# silu(G) * U: with |dG| <= GEMM_REL_TOL * max|G_row| and likewise for U (the
# GEMM bound), |d(silu(g) u)| <= |silu'(g)| |dg| |u| + |silu(g)| |du| + ...
# <= (1.1 + 1) * GEMM_REL_TOL * max|G_row| * max|U_row|, since
# silu'(g) lies in [-0.1, 1.1] and |silu(g)| <= |g|; the binary32 silu adds a
# few units of 2^-22 of |silu(g) u|.
SILU_MUL_REL_TOL = 2.2 * GEMM_REL_TOL


def silu_mul_ref(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """binary64 silu(g) * u = g / (1 + e^-g) * u."""
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g)) * u


def assert_silu_mul_close(y: np.ndarray, g: np.ndarray, u: np.ndarray, bf16: bool, what: str = ""):
    """y against silu(g) * u elementwise, g and u the binary64 GEMM references."""
    ref = silu_mul_ref(g, u)
    assert y.shape == ref.shape, (y.shape, ref.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    scale = np.max(np.abs(g), axis=1, keepdims=True) * np.max(np.abs(u), axis=1, keepdims=True)
    err = np.abs(y - ref)
    allow = SILU_MUL_REL_TOL * scale + (bf16_half_ulp(ref) if bf16 else 0.0)
    bad = err > allow
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = ", ".join(f"[{i},{j}] y={y[i, j]!r} ref={ref[i, j]!r}" for i, j in idx)
        raise AssertionError(f"{what}: {int(bad.sum())} elements outside tolerance; e.g. {detail}")
    with np.errstate(divide="ignore", invalid="ignore"):
        rel = np.where(scale > 0, np.max(np.maximum(err - (bf16_half_ulp(ref) if bf16 else 0.0), 0), axis=1,
                                         keepdims=True) / scale, 0.0)
    return float(np.max(rel)) if rel.size else 0.0
