"""Shared helpers of the GPU parity tests (comparison rules, randomized checks)."""
from __future__ import annotations

import numpy as np

from bit_quantized_tensor_gb300 import inputs

# Tolerance of every fp16-output path: relative Frobenius error <= 1e-3 and
# per-element |err| <= 1e-2 * (1 + |ref|), against the oracle's double result.
REL_FRO = 1e-3
ELEM_ABS = 1e-2


def assert_fp16_close(got_f16: np.ndarray, ref: np.ndarray, what: str = "") -> dict:
    got = got_f16.astype(np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = got - ref
    denom = np.linalg.norm(ref)
    rel = float(np.linalg.norm(err) / denom) if denom > 0 else float(np.linalg.norm(err))
    bound = ELEM_ABS * (1.0 + np.abs(ref))
    worst = float(np.max(np.abs(err) / bound)) if err.size else 0.0
    assert rel <= REL_FRO, f"{what}: relative Frobenius error {rel:.3e} > {REL_FRO}"
    assert worst <= 1.0, f"{what}: element error {worst:.3f} x allowed"
    return {"rel_fro": rel, "worst_elem_ratio": worst}


def freivalds_int(A: np.ndarray, B: np.ndarray, C: np.ndarray, trials: int = 3, seed: int = 99):
    """Check C == A . B^T (A: M x K, B: N x K integer values) with random
    vectors r in [-2^15, 2^15): C.r == A.(B^T.r), all in exact int64."""
    A64 = A.astype(np.int64)
    B64 = B.astype(np.int64)
    C64 = C.astype(np.int64)
    for t in range(trials):
        r = inputs.int_vector(B.shape[0], -(1 << 15), 1 << 15, seed + t)
        lhs = C64 @ r
        rhs = A64 @ (B64.T @ r)
        assert np.array_equal(lhs, rhs), f"Freivalds check failed on trial {t}"


def first_mismatch(got: np.ndarray, ref: np.ndarray) -> str:
    bad = np.argwhere(got != ref)
    if bad.size == 0:
        return "none"
    i, j = bad[0]
    return f"{len(bad)} mismatches, first at ({i},{j}): got {got[i, j]}, want {ref[i, j]}"
