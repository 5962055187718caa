"""Python binding of libnvfp4.so, the GB300 (sm_103a) NVFP4 linear-layer library.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels, called through its C ABI (include/nvfp4.h) with ctypes.  PyTorch
provides device memory and the current stream.  The functions carry the C
names; the ones that allocate their outputs with torch and return them are
thin conveniences over the same calls.

There is no CPU fallback: if libnvfp4.so is missing or cannot run on the
current device, every call raises.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import re
from typing import Optional

import torch

__all__ = [
    "NVFP4Error", "NVFP4Weight", "NVFP4Act", "lib", "library_path", "declared_functions",
    "nvfp4_scales_mma_bytes", "nvfp4_workspace_bytes", "nvfp4_quantize_fos", "nvfp4_quantize_act",
    "nvfp4_gemm_w4a16", "nvfp4_gemm_w4a4", "nvfp4_linear", "nvfp4_linear_silu_mul", "nvfp4_linear_noalloc",
    "nvfp4_dequantize", "nvfp4_qat_backward", "nvfp4_gptq_fos", "nvfp4_set_crossover",
    "nvfp4_get_crossover", "nvfp4_set_w4a16_rf_max_m", "nvfp4_get_w4a16_rf_max_m",
    "nvfp4_set_w4a16_sk_max_m", "nvfp4_get_w4a16_sk_max_m", "nvfp4_set_weight_prefetch",
    "nvfp4_get_weight_prefetch", "nvfp4_set_w4a4_cluster", "nvfp4_get_w4a4_cluster", "nvfp4_set_act_fos", "nvfp4_get_act_fos", "nvfp4_get_device_status", "nvfp4_measure_fp4_mma",
    "nvfp4_set_single_launch_quantizer", "nvfp4_get_single_launch_quantizer",
    "nvfp4_selftest_wait_timeout",
    "nvfp4_status_string",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_PKG)
library_path = os.path.join(_PKG, "libnvfp4.so")
header_path = os.path.join(_ROOT, "include", "nvfp4.h")

OK = 0
ERR_INVALID_ARG, ERR_SHAPE, ERR_ALIGN, ERR_WORKSPACE = 1, 2, 3, 4
ERR_NONFINITE, ERR_TIMEOUT, ERR_CUDA, ERR_UNSUPPORTED = 5, 6, 7, 8
OUT_BF16, OUT_F32 = 0, 1
OP_QUANTIZE_FOS, OP_QUANTIZE_ACT, OP_GEMM_W4A16, OP_GEMM_W4A4, OP_LINEAR, OP_LINEAR_SILU_MUL, OP_QAT_BACKWARD, \
    OP_GPTQ_FOS = 0, 1, 2, 3, 4, 5, 6, 7
DEFAULT_DIVISOR = 2688.0


class NVFP4Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


class _Weight(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales_mma", ctypes.c_void_p),
                ("tensor_scale", ctypes.c_void_p), ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise ImportError(f"{library_path} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(library_path)
        vp, i64, sz, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
        st = ctypes.c_int
        wp = ctypes.POINTER(_Weight)
        sig = {
            "nvfp4_scales_mma_bytes": (sz, [i64, i64]),
            "nvfp4_workspace_bytes": (sz, [ctypes.c_int, i64, i64, i64]),
            "nvfp4_quantize_fos": (st, [vp, i64, i64, f32, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
            "nvfp4_quantize_act": (st, [vp, i64, i64, f32, vp, vp, vp, vp, vp, sz, vp]),
            "nvfp4_gemm_w4a16": (st, [vp, i64, wp, vp, ctypes.c_int, vp, sz, vp]),
            "nvfp4_gemm_w4a4": (st, [vp, vp, vp, i64, wp, vp, ctypes.c_int, vp, sz, vp]),
            "nvfp4_linear": (st, [vp, i64, wp, vp, ctypes.c_int, vp, sz, vp]),
            "nvfp4_linear_noalloc": (st, [vp, i64, wp, vp, ctypes.c_int, vp]),
            "nvfp4_linear_silu_mul": (st, [vp, i64, wp, vp, ctypes.c_int, vp, sz, vp]),
            "nvfp4_dequantize": (st, [vp, vp, vp, i64, i64, vp, vp]),
            "nvfp4_gptq_fos": (st, [vp, i64, i64, vp, ctypes.c_float, vp, vp, vp, vp, vp, sz, vp]),
            "nvfp4_qat_backward": (st, [vp, i64, wp, vp, vp, vp, vp, vp, vp, sz, vp]),
            "nvfp4_set_crossover": (st, [i64, i64, i64]),
            "nvfp4_get_crossover": (i64, [i64, i64]),
            "nvfp4_set_w4a16_rf_max_m": (st, [i64]),
            "nvfp4_get_w4a16_rf_max_m": (i64, []),
            "nvfp4_set_w4a16_sk_max_m": (st, [i64]),
            "nvfp4_get_w4a16_sk_max_m": (i64, []),
            "nvfp4_set_weight_prefetch": (st, [ctypes.c_int]),
            "nvfp4_get_weight_prefetch": (ctypes.c_int, []),
            "nvfp4_set_w4a4_cluster": (st, [ctypes.c_int]),
            "nvfp4_set_act_fos": (st, [ctypes.c_int]),
            "nvfp4_get_act_fos": (ctypes.c_int, []),
            "nvfp4_get_w4a4_cluster": (ctypes.c_int, []),
            "nvfp4_set_single_launch_quantizer": (st, [ctypes.c_int]),
            "nvfp4_get_single_launch_quantizer": (ctypes.c_int, []),
            "nvfp4_get_device_status": (st, [vp]),
            "nvfp4_selftest_wait_timeout": (st, [vp]),
            "nvfp4_measure_fp4_mma": (st, [ctypes.c_int, vp, ctypes.c_int, ctypes.POINTER(ctypes.c_int), vp]),
            "nvfp4_status_string": (ctypes.c_char_p, [st]),
            "nvfp4_last_error": (ctypes.c_char_p, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def declared_functions() -> list:
    """Names of the functions include/nvfp4.h declares."""
    with open(header_path) as f:
        text = f.read()
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(nvfp4_\w+)\s*\(", text, flags=re.M)))


def _check(status: int, what: str):
    if status != OK:
        msg = lib().nvfp4_last_error().decode(errors="replace")
        raise NVFP4Error(status, f"{what}: {msg or nvfp4_status_string(status)}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _require_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def nvfp4_status_string(status: int) -> str:
    return lib().nvfp4_status_string(status).decode()


def nvfp4_scales_mma_bytes(rows: int, K: int) -> int:
    return lib().nvfp4_scales_mma_bytes(rows, K)


def nvfp4_workspace_bytes(op: int, M: int, N: int, K: int) -> int:
    return lib().nvfp4_workspace_bytes(op, M, N, K)


def nvfp4_set_crossover(N: int, K: int, m_threshold: int) -> None:
    _check(lib().nvfp4_set_crossover(N, K, m_threshold), "nvfp4_set_crossover")


def nvfp4_get_crossover(N: int = 0, K: int = 0) -> int:
    return lib().nvfp4_get_crossover(N, K)


def nvfp4_set_w4a16_rf_max_m(m: int) -> None:
    """Largest M that nvfp4_gemm_w4a16 sends to its register-file kernel."""
    _check(lib().nvfp4_set_w4a16_rf_max_m(m), "nvfp4_set_w4a16_rf_max_m")


def nvfp4_get_w4a16_rf_max_m() -> int:
    return lib().nvfp4_get_w4a16_rf_max_m()


def nvfp4_set_w4a16_sk_max_m(m: int) -> None:
    """Largest M that nvfp4_gemm_w4a16 sends to its persistent split-K kernel."""
    _check(lib().nvfp4_set_w4a16_sk_max_m(m), "nvfp4_set_w4a16_sk_max_m")


def nvfp4_get_w4a16_sk_max_m() -> int:
    return lib().nvfp4_get_w4a16_sk_max_m()


def nvfp4_set_weight_prefetch(enable: bool) -> None:
    """Let GEMM kernels read static weights before the previous kernel ends."""
    _check(lib().nvfp4_set_weight_prefetch(1 if enable else 0), "nvfp4_set_weight_prefetch")


def nvfp4_get_weight_prefetch() -> bool:
    return bool(lib().nvfp4_get_weight_prefetch())


def nvfp4_set_w4a4_cluster(ctas: int) -> None:
    """CTAs per cluster of the W4A4 kernel above 128 tokens: 2 or 1."""
    _check(lib().nvfp4_set_w4a4_cluster(ctas), "nvfp4_set_w4a4_cluster")


def nvfp4_get_w4a4_cluster() -> int:
    return lib().nvfp4_get_w4a4_cluster()


def nvfp4_set_act_fos(enable: bool) -> None:
    """nvfp4_linear's W4A4 branch: FourOverSix (True) or M=6-only (False) activations."""
    _check(lib().nvfp4_set_act_fos(1 if enable else 0), "nvfp4_set_act_fos")


def nvfp4_get_act_fos() -> bool:
    return bool(lib().nvfp4_get_act_fos())


def nvfp4_get_device_status(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device status word."""
    return lib().nvfp4_get_device_status(_stream(stream))


def nvfp4_selftest_wait_timeout(stream=None) -> None:
    """Launch the bounded-wait self-test (nvfp4_selftest_wait_timeout); the
    next nvfp4_get_device_status() returns ERR_TIMEOUT."""
    _check(lib().nvfp4_selftest_wait_timeout(_stream(stream)), "nvfp4_selftest_wait_timeout")


def nvfp4_set_single_launch_quantizer(enable: bool) -> None:
    """One cooperative launch per quantised tensor (True) or two launches."""
    _check(lib().nvfp4_set_single_launch_quantizer(1 if enable else 0), "nvfp4_set_single_launch_quantizer")


def nvfp4_get_single_launch_quantizer() -> bool:
    return bool(lib().nvfp4_get_single_launch_quantizer())


def nvfp4_measure_fp4_mma(iters: int = 20000, stream=None) -> dict:
    """Time the block-scaled FP4 MMA stream (nvfp4_measure_fp4_mma): one
    CTA pair per two SMs, iters x 4 MMAs of 256 x 256 x 64 each; returns the
    rate in TFLOP/s, the pairs launched and the median SM clock it implies."""
    dev = torch.device("cuda", torch.cuda.current_device())
    max_pairs = torch.cuda.get_device_properties(dev).multi_processor_count
    cycles = torch.zeros(max_pairs, dtype=torch.int64, device=dev)
    pairs = ctypes.c_int(0)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    _check(lib().nvfp4_measure_fp4_mma(iters, cycles.data_ptr(), max_pairs, ctypes.byref(pairs), s.cuda_stream),
           "nvfp4_measure_fp4_mma")
    e1.record(s)
    e1.synchronize()
    t = e0.elapsed_time(e1) * 1e-3
    flops = pairs.value * iters * 4 * 2.0 * 256 * 256 * 64
    cyc = cycles[: pairs.value].cpu().double()
    return {"tflops": flops / t / 1e12, "pairs": pairs.value, "seconds": t,
            "sm_mhz": float(cyc.median()) / t / 1e6 if pairs.value else 0.0}


@dataclasses.dataclass
class NVFP4Weight:
    """A quantised weight [N, K]: device tensors owned by torch."""
    codes: torch.Tensor            # uint8 [N, K/2]
    scales_mma: torch.Tensor       # uint8, MMA tiling
    tensor_scale: torch.Tensor     # float32 [1]
    N: int
    K: int
    scales: Optional[torch.Tensor] = None     # uint8 [N, K/16] logical
    choice: Optional[torch.Tensor] = None     # uint8 [N, K/16], 1 = M=4
    m4_count: Optional[torch.Tensor] = None   # int64 [1]

    def descriptor(self) -> _Weight:
        return _Weight(self.codes.data_ptr(), self.scales_mma.data_ptr(), self.tensor_scale.data_ptr(),
                       self.N, self.K)


@dataclasses.dataclass
class NVFP4Act:
    """Quantised activations [M, K]."""
    codes: torch.Tensor
    scales_mma: torch.Tensor
    tensor_scale: torch.Tensor
    M: int
    K: int
    scales: Optional[torch.Tensor] = None


def _workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def nvfp4_quantize_fos(W: torch.Tensor, divisor: float = 0.0, *, logical_scales: bool = True,
                       choice: bool = True, workspace: Optional[torch.Tensor] = None,
                       stream=None) -> NVFP4Weight:
    """FourOverSix NVFP4 quantisation of a bf16 weight [N, K] (nvfp4_quantize_fos)."""
    _require_cuda(W)
    if W.dtype != torch.bfloat16 or W.dim() != 2:
        raise ValueError("W must be a 2-D bfloat16 tensor")
    N, K = W.shape
    dev = W.device
    codes = torch.empty((N, K // 2), dtype=torch.uint8, device=dev)
    smma = torch.empty(max(nvfp4_scales_mma_bytes(N, K), 1), dtype=torch.uint8, device=dev)
    scales = torch.empty((N, K // 16), dtype=torch.uint8, device=dev) if logical_scales else None
    ch = torch.empty((N, K // 16), dtype=torch.uint8, device=dev) if choice else None
    ts = torch.empty(1, dtype=torch.float32, device=dev)
    m4 = torch.empty(1, dtype=torch.int64, device=dev)
    ws_bytes = nvfp4_workspace_bytes(OP_QUANTIZE_FOS, 0, N, K)
    ws = workspace if workspace is not None else _workspace(ws_bytes, dev)
    _check(lib().nvfp4_quantize_fos(W.data_ptr(), N, K, divisor, codes.data_ptr(), _ptr(scales),
                                    smma.data_ptr(), ts.data_ptr(), _ptr(ch), m4.data_ptr(),
                                    ws.data_ptr(), ws.numel(), _stream(stream)), "nvfp4_quantize_fos")
    return NVFP4Weight(codes, smma, ts, N, K, scales, ch, m4)


def nvfp4_quantize_act(X: torch.Tensor, divisor: float = 0.0, *, logical_scales: bool = False,
                       workspace: Optional[torch.Tensor] = None, stream=None) -> NVFP4Act:
    """M=6 NVFP4 quantisation of bf16 activations [M, K] (nvfp4_quantize_act)."""
    _require_cuda(X)
    if X.dtype != torch.bfloat16 or X.dim() != 2:
        raise ValueError("X must be a 2-D bfloat16 tensor")
    M, K = X.shape
    dev = X.device
    codes = torch.empty((M, K // 2), dtype=torch.uint8, device=dev)
    smma = torch.empty(max(nvfp4_scales_mma_bytes(M, K), 1), dtype=torch.uint8, device=dev)
    scales = torch.empty((M, K // 16), dtype=torch.uint8, device=dev) if logical_scales else None
    ts = torch.empty(1, dtype=torch.float32, device=dev)
    ws = workspace if workspace is not None else _workspace(nvfp4_workspace_bytes(OP_QUANTIZE_ACT, M, 0, K), dev)
    _check(lib().nvfp4_quantize_act(X.data_ptr(), M, K, divisor, codes.data_ptr(), _ptr(scales),
                                    smma.data_ptr(), ts.data_ptr(), ws.data_ptr(), ws.numel(),
                                    _stream(stream)), "nvfp4_quantize_act")
    return NVFP4Act(codes, smma, ts, M, K, scales)


def _out(M, N, out_dtype, dev, out):
    if out is not None:
        return out
    return torch.empty((M, N), dtype=torch.float32 if out_dtype == OUT_F32 else torch.bfloat16, device=dev)


def nvfp4_gemm_w4a16(X: torch.Tensor, W: NVFP4Weight, out_dtype: int = OUT_BF16,
                     out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    _require_cuda(X, out)
    M = X.shape[0]
    Y = _out(M, W.N, out_dtype, X.device, out)
    d = W.descriptor()
    _check(lib().nvfp4_gemm_w4a16(X.data_ptr(), M, ctypes.byref(d), Y.data_ptr(), out_dtype, None, 0,
                                  _stream(stream)), "nvfp4_gemm_w4a16")
    return Y


def nvfp4_gemm_w4a4(A: NVFP4Act, W: NVFP4Weight, out_dtype: int = OUT_BF16,
                    out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    _require_cuda(out)
    Y = _out(A.M, W.N, out_dtype, A.codes.device, out)
    d = W.descriptor()
    _check(lib().nvfp4_gemm_w4a4(A.codes.data_ptr(), A.scales_mma.data_ptr(), A.tensor_scale.data_ptr(), A.M,
                                 ctypes.byref(d), Y.data_ptr(), out_dtype, None, 0, _stream(stream)),
           "nvfp4_gemm_w4a4")
    return Y


def nvfp4_linear(X: torch.Tensor, W: NVFP4Weight, out_dtype: int = OUT_BF16,
                 out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                 stream=None) -> torch.Tensor:
    """Y = X W^T with the M-based W4A16 / W4A4 dispatch (nvfp4_linear)."""
    _require_cuda(X, out)
    M = X.shape[0]
    Y = _out(M, W.N, out_dtype, X.device, out)
    ws = workspace if workspace is not None else _workspace(nvfp4_workspace_bytes(OP_LINEAR, M, W.N, W.K),
                                                            X.device)
    d = W.descriptor()
    _check(lib().nvfp4_linear(X.data_ptr(), M, ctypes.byref(d), Y.data_ptr(), out_dtype, ws.data_ptr(),
                              ws.numel(), _stream(stream)), "nvfp4_linear")
    return Y


def nvfp4_linear_silu_mul(X: torch.Tensor, W: NVFP4Weight, out_dtype: int = OUT_BF16,
                          out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                          stream=None) -> torch.Tensor:
    """Y = silu(X W_gate^T) * (X W_up^T) for a gate/up weight [2F, K] (nvfp4_linear_silu_mul)."""
    _require_cuda(X, out)
    M = X.shape[0]
    Y = _out(M, W.N // 2, out_dtype, X.device, out)
    ws = workspace if workspace is not None else _workspace(
        nvfp4_workspace_bytes(OP_LINEAR_SILU_MUL, M, W.N, W.K), X.device)
    d = W.descriptor()
    _check(lib().nvfp4_linear_silu_mul(X.data_ptr(), M, ctypes.byref(d), Y.data_ptr(), out_dtype, ws.data_ptr(),
                                       ws.numel(), _stream(stream)), "nvfp4_linear_silu_mul")
    return Y


NOALLOC_SCRATCH_BYTES = 32 << 20


def nvfp4_linear_noalloc(X: torch.Tensor, W: NVFP4Weight, out_dtype: int = OUT_BF16,
                         out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """nvfp4_linear with the library's built-in scratch instead of a workspace,
    for callers that cannot allocate device memory (the output tensor is still
    the caller's)."""
    _require_cuda(X, out)
    M = X.shape[0]
    Y = _out(M, W.N, out_dtype, X.device, out)
    d = W.descriptor()
    _check(lib().nvfp4_linear_noalloc(X.data_ptr(), M, ctypes.byref(d), Y.data_ptr(), out_dtype,
                                      _stream(stream)), "nvfp4_linear_noalloc")
    return Y


def nvfp4_dequantize(codes: torch.Tensor, scales_mma: torch.Tensor, tensor_scale: torch.Tensor, rows: int, K: int,
                     out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """NVFP4 [rows, K] -> bf16 [rows, K] (nvfp4_dequantize)."""
    _require_cuda(codes, out)
    Y = out if out is not None else torch.empty((rows, K), dtype=torch.bfloat16, device=codes.device)
    _check(lib().nvfp4_dequantize(codes.data_ptr(), scales_mma.data_ptr(), tensor_scale.data_ptr(), rows, K,
                                  Y.data_ptr(), _stream(stream)), "nvfp4_dequantize")
    return Y


def nvfp4_qat_backward(dY: torch.Tensor, W: NVFP4Weight, A: Optional[NVFP4Act], want_dx: bool = True,
                       want_dw: bool = True, stream=None):
    """(dX bf16 [M, K], dW fp32 [N, K]) of the FP4-forward linear Y = X_hat W_hat^T
    with straight-through gradients (nvfp4_qat_backward); None for a skipped one."""
    _require_cuda(dY)
    M = dY.shape[0]
    dev = dY.device
    dX = torch.empty((M, W.K), dtype=torch.bfloat16, device=dev) if want_dx else None
    dW = torch.empty((W.N, W.K), dtype=torch.float32, device=dev) if want_dw else None
    ws = _workspace(nvfp4_workspace_bytes(OP_QAT_BACKWARD, M, W.N, W.K), dev)
    d = W.descriptor()
    _check(lib().nvfp4_qat_backward(dY.data_ptr(), M, ctypes.byref(d),
                                    A.codes.data_ptr() if A is not None else None,
                                    A.scales_mma.data_ptr() if A is not None else None,
                                    A.tensor_scale.data_ptr() if A is not None else None,
                                    dX.data_ptr() if dX is not None else None,
                                    dW.data_ptr() if dW is not None else None, ws.data_ptr(), ws.numel(),
                                    _stream(stream)), "nvfp4_qat_backward")
    return dX, dW


def nvfp4_gptq_fos(W: torch.Tensor, H: torch.Tensor, damp: float = 0.01, stream=None) -> NVFP4Weight:
    """GPTQ inside FourOverSix scales (nvfp4_gptq_fos): W bf16 [N, K], H fp32 [K, K]."""
    _require_cuda(W, H)
    if W.dtype != torch.bfloat16 or W.dim() != 2 or H.dtype != torch.float32 or not H.is_contiguous():
        raise ValueError("W must be a 2-D bfloat16 tensor and H a contiguous float32 [K, K] tensor")
    N, K = W.shape
    dev = W.device
    codes = torch.empty((N, K // 2), dtype=torch.uint8, device=dev)
    scales = torch.empty((N, K // 16), dtype=torch.uint8, device=dev)
    smma = torch.empty(nvfp4_scales_mma_bytes(N, K), dtype=torch.uint8, device=dev)
    ts = torch.empty(1, dtype=torch.float32, device=dev)
    ws = _workspace(nvfp4_workspace_bytes(OP_GPTQ_FOS, 0, N, K), dev)
    _check(lib().nvfp4_gptq_fos(W.contiguous().data_ptr(), N, K, H.data_ptr(), float(damp), codes.data_ptr(),
                                scales.data_ptr(), smma.data_ptr(), ts.data_ptr(), ws.data_ptr(), ws.numel(),
                                _stream(stream)), "nvfp4_gptq_fos")
    return NVFP4Weight(codes=codes, scales_mma=smma, tensor_scale=ts, N=N, K=K, scales=scales)
