"""Numerical arguments behind two readings of the W4A4 page (CPU, numpy).

The page writes Y = (Q(X).Q(W)^T) (.) scale with block-wise K scales.  A
tensor-core design can either keep each 64-wide block's integer partial
exact and apply sX * sW afterwards (what the library does), or fold the
scales into the MMA operands (q * s rounded to the operand type) and let one
accumulation run over all of K.  The fold is faster but rounds every operand;
the tests below show that on the workload's distributions (X, W ~ N(0, 1),
symmetric absmax codes with fp16 scales) every fold misses the per-element
tolerance 1e-2 (1 + |ref|), while the exact-partial form meets it by
construction.  The options are the fp16 fold (one fp16 operand per side) and
the two-term e4m3 split of q * s (hi + lo per side, the cross products as
extra K columns of an fp8 MMA).
"""
import numpy as np


def _e4m3(x):
    """Round to nearest even onto e4m3 (bias 7, 3 mantissa bits, max 448,
    subnormal step 2^-9)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    e = np.maximum(np.floor(np.log2(np.where(a > 0, a, 1.0))), -6.0)
    step = 2.0 ** (e - 3)
    return np.sign(x) * np.minimum(np.round(a / step) * step, 448.0)


def _quantize(X, blk=64):
    M, K = X.shape
    Xb = X.reshape(M, K // blk, blk)
    s = (np.abs(Xb).max(axis=2) / np.float32(7.0)).astype(np.float32).astype(np.float16)
    sf = s.astype(np.float32)[..., None]
    q = np.where(sf > 0, np.clip(np.rint(Xb / np.where(sf > 0, sf, 1)), -8, 7), 0)
    return q.reshape(M, K), s.astype(np.float64)


def _worst_ratio(K, fold, M=32, N=128):
    rng = np.random.default_rng(11)
    X = rng.standard_normal((M, K)).astype(np.float32)
    W = rng.standard_normal((N, K)).astype(np.float32)
    qx, sx = _quantize(X)
    qw, sw = _quantize(W)
    a = qx * np.repeat(sx, 64, axis=1)   # q * s exactly (double)
    b = qw * np.repeat(sw, 64, axis=1)
    ref = a @ b.T
    return np.max(np.abs(fold(a, b) - ref) / (1e-2 * (1 + np.abs(ref))))


def _fp16_fold(a, b):
    return a.astype(np.float16).astype(np.float64) @ b.astype(np.float16).astype(np.float64).T


def _e4m3_split(a, b):
    ah, bh = _e4m3(a), _e4m3(b)
    al, bl = _e4m3(a - ah), _e4m3(b - bh)
    return ah @ bh.T + ah @ bl.T + al @ bh.T


def test_e4m3_matches_the_format_on_known_values():
    assert list(_e4m3([1.0, -8.0, 448.0, 1000.0, 2.0 ** -9, 1.0625, 1.1875])) == \
        [1.0, -8.0, 448.0, 448.0, 2.0 ** -9, 1.0, 1.25]


def test_every_operand_fold_misses_the_per_element_bound():
    # 64K outputs at K = 256 (a short K hides the error in few samples), 4K at 8192
    for K, M, N in ((256, 128, 512), (8192, 32, 128)):
        assert _worst_ratio(K, _fp16_fold, M, N) > 1.0, K
        assert _worst_ratio(K, _e4m3_split, M, N) > 2.0, K


def test_the_exact_block_partial_form_meets_it():
    # the block partials are exact integers; applying sX * sW in fp32 and
    # accumulating 128 blocks in fp32 leaves only fp32 rounding
    def exact_partials(a, b):
        K = a.shape[1]
        y = np.zeros((a.shape[0], b.shape[0]), dtype=np.float32)
        for j in range(K // 64):
            y += (a[:, 64 * j:64 * j + 64] @ b[:, 64 * j:64 * j + 64].T).astype(np.float32)
        return y.astype(np.float64)
    assert _worst_ratio(8192, exact_partials) < 0.05
