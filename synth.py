"""Seeded synthetic inputs for the NVFP4 linear-layer workloads.

This module only draws random numbers and rounds them to bfloat16; it holds
none of the quantiser's or the GEMMs' arithmetic.  Both the CPU oracle and the
CUDA library are fed from here, so they see identical bits.

Every generator uses numpy's ``Generator(PCG64(seed))``, draws in float32,
applies the workload's modifications, then rounds to bf16 (round to nearest,
ties to even) and returns the raw uint16 bit patterns.

The pages measure on real MiniCPM-SALA weights and contest prompts, which are
not available; these LLM-shaped tensors stand in for them.
"""
from __future__ import annotations

import numpy as np


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def weight_normal(N: int, K: int, seed: int, std: float = 0.02, outlier_frac: float = 0.0,
                  outlier_mult: float = 8.0) -> np.ndarray:
    """W [N, K] ~ N(0, std^2); exactly round(outlier_frac*N*K) entries, at
    positions drawn uniformly without replacement, are multiplied by
    ``outlier_mult``."""
    rng = _rng(seed)
    w = rng.standard_normal((N, K), dtype=np.float32) * np.float32(std)
    n_out = int(round(outlier_frac * N * K))
    if n_out:
        pos = rng.choice(N * K, size=n_out, replace=False)
        w.reshape(-1)[pos] *= np.float32(outlier_mult)
    return f32_to_bf16_bits(w)


def weight_lognormal_rows(N: int, K: int, seed: int, std: float = 0.02,
                          sigma: float = 0.5) -> np.ndarray:
    """W [N, K] ~ N(0, (std * f_n)^2) with a per-output-row factor
    f_n ~ LogNormal(0, sigma), so blocks have varied dynamic range."""
    rng = _rng(seed)
    f = rng.lognormal(0.0, sigma, size=(N, 1)).astype(np.float32)
    w = rng.standard_normal((N, K), dtype=np.float32) * np.float32(std) * f
    return f32_to_bf16_bits(w)


def act_normal(M: int, K: int, seed: int) -> np.ndarray:
    """Activations X [M, K] ~ N(0, 1)."""
    return f32_to_bf16_bits(_rng(seed).standard_normal((M, K), dtype=np.float32))


def act_student_t(M: int, K: int, seed: int, nu: float = 4.0, scale: float = 0.5) -> np.ndarray:
    """Activations X [M, K] ~ scale * Student-t(nu) (heavy-tailed, prefill-like)."""
    x = _rng(seed).standard_t(nu, size=(M, K)).astype(np.float32) * np.float32(scale)
    return f32_to_bf16_bits(x)


# --------------------------------------------------------------- workloads ---
# Seeds: the tiny case uses seed 0 for W and 1 for x; the others use
# 100 * workload + tensor index.

def tiny_case():
    """256 x 512 weight, N(0, 0.02^2) with 1% outliers x8; x [1, 512] ~ N(0,1)."""
    return weight_normal(256, 512, seed=0, outlier_frac=0.01), act_normal(1, 512, seed=1)


DECODE_M = (1, 2, 4, 8, 16, 32, 48)
MLP_M = (1, 8, 32, 48)
PREFILL_M = (64, 256, 1024, 4096, 16384)


def decode_weight():
    """Decode-shaped linear: W [4096, 4096], N(0, 0.02^2), 0.5% outliers x8."""
    return weight_normal(4096, 4096, seed=200, outlier_frac=0.005)


def decode_act(M: int):
    return act_normal(M, 4096, seed=201 + M)


def mlp_weights():
    """MLP-shaped linears: gate/up [2*11008, 4096] and down [4096, 11008],
    row std multiplied by LogNormal(0, 0.5)."""
    return (weight_lognormal_rows(2 * 11008, 4096, seed=300),
            weight_lognormal_rows(4096, 11008, seed=301))


def prefill_weight():
    """Prefill linear: W [11008, 4096], N(0, 0.02^2) with 1% outliers x8."""
    return weight_normal(11008, 4096, seed=400, outlier_frac=0.01)


def prefill_act(M: int):
    """Prefill activations [M, 4096] ~ 0.5 * Student-t(4)."""
    return act_student_t(M, 4096, seed=401 + M)


MODEL_LAYER_SHAPES = (("qkv", 6144, 4096), ("o", 4096, 4096), ("gate_up", 2 * 11008, 4096),
                      ("down", 4096, 11008))
MODEL_LAYERS = 32


def model_layer_weight(layer: int, which: int):
    """One matrix of the synthetic 32-layer stack, N(0, 0.02^2), 0.5% outliers x8."""
    _, N, K = MODEL_LAYER_SHAPES[which]
    return weight_normal(N, K, seed=500 + 4 * layer + which, outlier_frac=0.005)
