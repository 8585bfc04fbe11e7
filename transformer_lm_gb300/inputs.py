"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds input generation only (random numbers, shapes and the
initialisation recipe); none of the training step's arithmetic lives here.
Both the CUDA path and the CPU oracle receive exactly the arrays produced here.

Random numbers come from a counter-based generator: element ``i`` of stream
``s`` under seed ``seed`` is the SplitMix64 output function (Steele, Lea and
Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014) applied
to ``seed * 0x9E3779B97F4A7C15 + (s << 40) + i`` (mod 2**64). Uniforms take the
top 53 bits; normals use the Box-Muller transform on two consecutive uniforms.
All integer work is exact uint64 arithmetic, so every platform produces the
same bits.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


@dataclass(frozen=True)
class GPT2Dims:
    L: int
    C: int
    NH: int
    V: int
    Vp: int
    maxT: int


# the model shapes used by the tests and the benchmark
TINY = GPT2Dims(L=2, C=64, NH=4, V=512, Vp=512, maxT=32)
GPT2_124M = GPT2Dims(L=12, C=768, NH=12, V=50257, Vp=50304, maxT=1024)
GPT2_350M = GPT2Dims(L=24, C=1024, NH=16, V=50257, Vp=50304, maxT=1024)

PARAM_NAMES = ["wte", "wpe", "ln1w", "ln1b", "qkvw", "qkvb", "attprojw", "attprojb",
               "ln2w", "ln2b", "fcw", "fcb", "fcprojw", "fcprojb", "lnfw", "lnfb"]


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def random_u64(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    base = np.uint64((seed * 0x9E3779B97F4A7C15 + (stream << 40)) & 0xFFFFFFFFFFFFFFFF)
    idx = np.arange(start, start + n, dtype=np.uint64)
    return _mix(idx + base)


def uniform(seed: int, stream: int, n: int) -> np.ndarray:
    """Uniform float64 in the open interval (0, 1)."""
    z = random_u64(seed, stream, n)
    return ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)


def normal(seed: int, stream: int, n: int, std: float = 1.0) -> np.ndarray:
    """Standard normals (scaled by std) by Box-Muller, float64."""
    m = (n + 1) // 2
    u = uniform(seed, stream, 2 * m)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    out = np.empty(2 * m)
    out[0::2] = r * np.cos(2.0 * math.pi * u2)
    out[1::2] = r * np.sin(2.0 * math.pi * u2)
    return out[:n] * std


def tokens(seed: int, stream: int, B: int, T: int, V: int) -> np.ndarray:
    """Uniform int32 token ids in [0, V), shape (B, T)."""
    z = random_u64(seed, stream, B * T)
    return (z % np.uint64(V)).astype(np.int32).reshape(B, T)


def param_sizes(d: GPT2Dims) -> list[int]:
    C, L = d.C, d.L
    return [d.Vp * C, d.maxT * C, L * C, L * C, L * 3 * C * C, L * 3 * C, L * C * C, L * C,
            L * C, L * C, L * 4 * C * C, L * 4 * C, L * C * 4 * C, L * C, C, C]


def gpt2_params(d: GPT2Dims, seed: int, perturb: bool = False) -> np.ndarray:
    """Flat float32 parameters in the 16-tensor order.

    Recipe: every weight matrix and both embeddings ~ N(0, 0.02); the two
    residual out-projections (attprojw, fcprojw) ~ N(0, 0.02/sqrt(2L)); biases 0;
    LayerNorm gains 1 and biases 0; the padded rows [V, Vp) of wte are 0.
    ``perturb=True`` (used by parity tests so that every term is exercised)
    draws biases ~ N(0, 0.02), LayerNorm gains ~ 1 + N(0, 0.1) and LayerNorm
    biases ~ N(0, 0.02) instead.
    """
    sizes = param_sizes(d)
    resid_std = 0.02 / math.sqrt(2 * d.L) if d.L > 0 else 0.02
    parts = []
    for s, (name, n) in enumerate(zip(PARAM_NAMES, sizes)):
        if name in ("wte", "wpe", "qkvw", "fcw"):
            a = normal(seed, s, n, 0.02)
            if name == "wte":
                a = a.reshape(d.Vp, d.C)
                a[d.V:] = 0.0
                a = a.reshape(-1)
        elif name in ("attprojw", "fcprojw"):
            a = normal(seed, s, n, resid_std)
        elif name in ("ln1w", "ln2w", "lnfw"):
            a = 1.0 + (normal(seed, s, n, 0.1) if perturb else 0.0) * np.ones(n)
        else:  # biases and LayerNorm shifts
            a = normal(seed, s, n, 0.02) if perturb else np.zeros(n)
        parts.append(np.asarray(a, dtype=np.float32).reshape(-1))
    return np.concatenate(parts)


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) & np.uint64(0xFFFF0000)
    return u.astype(np.uint32).view(np.float32)


def round_to_fp16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest IEEE half (ties to even, numpy's
    conversion); returns float32."""
    return np.ascontiguousarray(a, dtype=np.float32).astype(np.float16).astype(np.float32)


def fused_op_inputs(M: int, K: int, N: int, seed: int):
    """x ~ N(0,1) (M,K); W ~ N(0, 1/sqrt(K)) (N,K) in nn.Linear layout; b ~ U(-0.1, 0.1)."""
    x = normal(seed, 100, M * K).astype(np.float32).reshape(M, K)
    W = normal(seed, 101, N * K, 1.0 / math.sqrt(K)).astype(np.float32).reshape(N, K)
    b = ((uniform(seed, 102, N) * 0.2) - 0.1).astype(np.float32)
    return x, W, b
