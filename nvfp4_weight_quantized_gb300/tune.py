"""Measure the W4A16 / W4A4 crossover of nvfp4_linear on the current GPU.

The dispatch rule ("SOAR 2026 Recap ...", section "1. Quantization and GEMM
dispatch") picks, per token count M, whichever of the two GEMM paths is faster;
the pages found the curves crossing near M = 48 on their GPU.  This module
times both paths for one weight shape with CUDA graphs (many launches per
replay, weights rotated so reads are cold) and returns the largest M for which
W4A16 is still faster, optionally installing it with nvfp4_set_crossover.
"""
from __future__ import annotations

import torch

from . import (OUT_BF16, NVFP4Weight, lib, nvfp4_gemm_w4a16, nvfp4_gemm_w4a4, nvfp4_quantize_act,
               nvfp4_quantize_fos, nvfp4_set_crossover)

DEFAULT_SWEEP = (1, 2, 4, 8, 16, 24, 32, 48, 64, 96, 128, 192, 256)


def _time_graphs(fn, reps: int, nsets: int, stream) -> float:
    """Seconds per call of fn(i): nsets graphs of `reps` calls each (call i of
    set k gets index k * reps + i), replayed once to warm up, then timed as
    one pass over all sets, so that no call reuses what the previous replay
    left in L2 when the indexed data is larger than L2."""
    with torch.cuda.stream(stream):
        for i in range(2):
            fn(i)
    stream.synchronize()
    graphs = []
    for k in range(nsets):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(reps):
                fn(k * reps + i)
        graphs.append(g)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for g in graphs:
            g.replay()
        e0.record(stream)
        for g in graphs:
            g.replay()
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) * 1e-3 / (reps * nsets)


def _time_graph(fn, reps: int, stream) -> float:
    return _time_graphs(fn, reps, 1, stream)


def measure(N: int, K: int, sweep=DEFAULT_SWEEP, copies: int = 0, reps: int = 16, seed: int = 0):
    """Per-M seconds per call of both paths: {M: (t_w4a16, t_w4a4)}.  The
    weight is copied `copies` times (default: enough for twice the L2) and
    every timed call reads a different copy."""
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev).manual_seed(seed)
    w = (torch.randn(N, K, device=dev, generator=gen) * 0.02).to(torch.bfloat16)
    q = nvfp4_quantize_fos(w, logical_scales=False, choice=False)
    wbytes = N * K // 2 + N * K // 16
    if copies <= 0:
        copies = max(2 * reps, -(-2 * 126 * 2**20 // wbytes))
    nsets = max(1, -(-copies // reps))
    copies = nsets * reps
    Ws = [NVFP4Weight(q.codes.clone(), q.scales_mma.clone(), q.tensor_scale.clone(), N, K)
          for _ in range(copies)]
    stream = torch.cuda.Stream(device=dev)
    out = {}
    for M in sweep:
        x = torch.randn(M, K, device=dev, generator=gen).to(torch.bfloat16)
        y = torch.empty(M, N, device=dev, dtype=torch.bfloat16)
        a = nvfp4_quantize_act(x)
        ws = torch.empty(8192, dtype=torch.uint8, device=dev)

        def f16(i):
            nvfp4_gemm_w4a16(x, Ws[i % copies], OUT_BF16, out=y, stream=stream)

        def f4(i):  # online activation quantisation into preallocated buffers, then the GEMM
            st = lib().nvfp4_quantize_act(x.data_ptr(), M, K, 0.0, a.codes.data_ptr(), None,
                                          a.scales_mma.data_ptr(), a.tensor_scale.data_ptr(), ws.data_ptr(),
                                          ws.numel(), stream.cuda_stream)
            assert st == 0
            nvfp4_gemm_w4a4(a, Ws[i % copies], OUT_BF16, out=y, stream=stream)

        out[M] = (_time_graphs(f16, reps, nsets, stream), _time_graphs(f4, reps, nsets, stream))
    return out


def crossover_from(times: dict) -> int:
    """Largest M of the sweep for which W4A16 is at least as fast as W4A4,
    counting from the smallest M until W4A4 is faster twice in a row."""
    best = 0
    losses = 0
    for M in sorted(times):
        t16, t4 = times[M]
        if t16 <= t4:
            best = M
            losses = 0
        else:
            losses += 1
            if losses >= 2:
                break
    return best


def tune(N: int, K: int, install: bool = True, **kw) -> int:
    times = measure(N, K, **kw)
    m = crossover_from(times)
    if install:
        nvfp4_set_crossover(N, K, m)
    return m
