"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module only draws random numbers with numpy's PCG64 generator; it holds
none of the quantized-GEMM arithmetic.  A uniformly random byte is exactly a
pair of independent signed 4-bit values uniform over [-8, 7], so packed INT4
operands are drawn as random bytes.

Seeds follow one convention everywhere: ``1000 + workload index`` for the
left operand (A / X), ``2000 + index`` for the right operand (B / W) and
``3000 + index`` for scales, low-rank factors and bias.
"""
from __future__ import annotations

import numpy as np

# Workload table.  Index = position in this list (also the seed offset).
WORKLOADS = [
    {"name": "int8_gemm_512", "op": "qgemm_s8", "M": 512, "N": 512, "K": 512},
    {"name": "int4_gemm_2048", "op": "qgemm_s4", "M": 2048, "N": 2048, "K": 2048},
    {"name": "sweep", "ops": ["qgemm_s8", "qgemm_s4", "gemm_f16"],
     "sizes": [512, 1024, 2048, 4096, 8192]},
    {"name": "w4a16_4096", "op": "w4a16_gemm", "N": 4096, "K": 4096, "Ms": [1, 16, 128],
     "group": 128},
    {"name": "w4a4_lowrank", "op": "w4a4_gemm", "M": 4096, "N": 8192, "K": 8192,
     "rank": 32, "block": 64},
]


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def s8_uniform(rows: int, cols: int, seed: int) -> np.ndarray:
    """int8 matrix, i.i.d. uniform over [-128, 127]."""
    return rng(seed).integers(-128, 128, size=(rows, cols), dtype=np.int8)


def s8_in_range(rows: int, cols: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """int8 matrix, i.i.d. uniform over [lo, hi]."""
    return rng(seed).integers(lo, hi + 1, size=(rows, cols), dtype=np.int8)


def s4_packed_uniform(rows: int, K: int, seed: int) -> np.ndarray:
    """Packed signed 4-bit matrix (rows x K/2 bytes), values uniform over [-8, 7]."""
    if K % 2:
        raise ValueError("K must be even for packed 4-bit data")
    return rng(seed).integers(0, 256, size=(rows, K // 2), dtype=np.uint8)


def f16_normal(rows: int, cols: int, seed: int, sigma: float = 1.0) -> np.ndarray:
    """fp16 matrix, i.i.d. N(0, sigma^2) drawn in double then rounded to fp16."""
    return (rng(seed).standard_normal((rows, cols)) * sigma).astype(np.float16)


def f32_normal(rows: int, cols: int, seed: int, sigma: float = 1.0) -> np.ndarray:
    """fp32 matrix, i.i.d. N(0, sigma^2)."""
    return (rng(seed).standard_normal((rows, cols)) * sigma).astype(np.float32)


def f16_uniform(rows: int, cols: int, lo: float, hi: float, seed: int) -> np.ndarray:
    """fp16 matrix, i.i.d. uniform over [lo, hi) drawn in double, rounded to fp16."""
    return rng(seed).uniform(lo, hi, size=(rows, cols)).astype(np.float16)


def int_vector(n: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """int64 vector uniform over [lo, hi) (used for randomized product checks)."""
    return rng(seed).integers(lo, hi, size=n, dtype=np.int64)


def sample_rows(M: int, count: int, seed: int) -> np.ndarray:
    """Sorted distinct row indices in [0, M), always including the first and last row."""
    count = min(count, M)
    idx = set(rng(seed).choice(M, size=count, replace=False).tolist())
    idx.update({0, M - 1})
    return np.array(sorted(idx), dtype=np.int64)
