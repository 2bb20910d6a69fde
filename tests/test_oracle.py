"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test compares the oracle with a closed form, a hand-derived fixture
(tests/golden/), an invariant of the definition, or an independent library
routine (numpy's exact int64 / float64 matmul, numpy's float16 conversion),
chosen so that a dropped term, a wrong sign, a wrong index or a transposed
operand in the oracle fails at least one of them.
"""
import os

import numpy as np
import pytest

from bit_quantized_tensor_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- fp16 ----

def test_half_to_double_all_patterns(oracle):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.halves_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_float_to_half_matches_numpy_rounding(oracle):
    r = inputs.rng(7)
    vals = np.concatenate([
        r.standard_normal(3000).astype(np.float32) * np.float32(100),
        r.standard_normal(1000).astype(np.float32) * np.float32(1e-5),  # subnormal range
        np.array([1 + 2**-11, 1 + 3 * 2**-11, 65504, 65519, 65520, 1e9, -1e9, 0.0,
                  -0.0, 2**-25, 2**-24, 1.5 * 2**-24, 2.5 * 2**-24], dtype=np.float32),
    ])
    got = np.array([oracle.float_to_half(float(v)) for v in vals], dtype=np.uint16)
    ref = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def test_double_to_half_single_rounding(oracle):
    # 1 + 2^-11 + 2^-30 is just above the tie: one rounding gives 1 + 2^-10;
    # rounding to binary32 first would give the tie 1 + 2^-11 and then 1.0.
    x = 1 + 2**-11 + 2**-30
    assert oracle.double_to_half(x) == np.float16(1 + 2**-10).view(np.uint16)


# -------------------------------------------------------------- packing ----

def _golden_nibbles():
    rows = []
    with open(os.path.join(GOLDEN, "s4_nibbles.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                b, lo, hi = line.split()
                rows.append((int(b, 16), int(lo), int(hi)))
    return rows


def test_s4_unpack_golden(oracle):
    rows = _golden_nibbles()
    P = np.array([[b for b, _, _ in rows]], dtype=np.uint8)
    V = oracle.s4_unpack(P, 2 * len(rows))
    expect = np.array([[v for _, lo, hi in rows for v in (lo, hi)]], dtype=np.int8)
    assert np.array_equal(V, expect)


def test_s4_round_trip_all_bytes(oracle):
    P = np.arange(256, dtype=np.uint8).reshape(1, 256)
    V = oracle.s4_unpack(P, 512)
    assert V.min() == -8 and V.max() == 7
    assert np.array_equal(oracle.s4_pack(V), P)
    # every (even, odd) pair of values occurs exactly once
    pairs = {(int(V[0, 2 * i]), int(V[0, 2 * i + 1])) for i in range(256)}
    assert len(pairs) == 256


def test_s4_pack_rejects_out_of_range(oracle):
    with pytest.raises(ValueError):
        oracle.s4_pack(np.array([[8, 0]], dtype=np.int8))


# ------------------------------------------------------------- INT8 GEMM ----

@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (17, 9, 33), (64, 48, 80)])
def test_gemm_s8_matches_numpy_int64(oracle, M, N, K):
    A = inputs.s8_uniform(M, K, 11 + M)
    B = inputs.s8_uniform(N, K, 12 + N)
    C = oracle.gemm_s8(A, B)
    ref = A.astype(np.int64) @ B.astype(np.int64).T
    assert C.dtype == np.int32
    assert np.array_equal(C.astype(np.int64), ref)


@pytest.mark.parametrize("K", [16, 1024, 8192])
def test_gemm_s8_closed_form_extremes(oracle, K):
    A = np.full((2, K), -128, dtype=np.int8)
    B = np.full((3, K), -128, dtype=np.int8)
    assert np.all(oracle.gemm_s8(A, B) == 16384 * K)
    B2 = np.full((3, K), 127, dtype=np.int8)
    assert np.all(oracle.gemm_s8(A, B2) == -16256 * K)


def test_gemm_s8_identity_gives_transpose(oracle):
    K, N = 24, 10
    A = np.eye(K, dtype=np.int8)
    B = inputs.s8_uniform(N, K, 5)
    assert np.array_equal(oracle.gemm_s8(A, B), B.T.astype(np.int32))


def test_gemm_s8_ones_gives_row_sums(oracle):
    K, N = 40, 6
    A = np.ones((3, K), dtype=np.int8)
    B = inputs.s8_uniform(N, K, 6)
    sums = B.astype(np.int64).sum(axis=1)
    assert np.array_equal(oracle.gemm_s8(A, B), np.tile(sums, (3, 1)).astype(np.int32))


def test_gemm_s8_transpose_invariant(oracle):
    A = inputs.s8_uniform(13, 21, 8)
    B = inputs.s8_uniform(7, 21, 9)
    assert np.array_equal(oracle.gemm_s8(A, B), oracle.gemm_s8(B, A).T)


def test_gemm_s8_linear_in_A(oracle):
    A1 = inputs.s8_in_range(9, 30, -60, 60, 10)
    A2 = inputs.s8_in_range(9, 30, -60, 60, 11)
    B = inputs.s8_uniform(5, 30, 12)
    lhs = oracle.gemm_s8((A1.astype(np.int16) + A2).astype(np.int8), B)
    assert np.array_equal(lhs, oracle.gemm_s8(A1, B) + oracle.gemm_s8(A2, B))


def test_gemm_s8_detects_int32_overflow(oracle):
    K = 131072  # 16384 * 131072 = 2^31 > INT32_MAX
    A = np.full((1, K), -128, dtype=np.int8)
    with pytest.raises(ValueError):
        oracle.gemm_s8(A, A)


def test_gemm_s8_leading_dimension(oracle):
    import ctypes
    lib = oracle._load()
    M, N, K, ld = 4, 3, 5, 9
    Ap = inputs.s8_uniform(M, ld, 13)
    Bp = inputs.s8_uniform(N, ld, 14)
    C = np.zeros((M, 7), dtype=np.int32)
    rc = lib.orc_gemm_s8(M, N, K, Ap.ctypes.data, ld, Bp.ctypes.data, ld, C.ctypes.data, 7)
    assert rc == 0
    ref = Ap[:, :K].astype(np.int64) @ Bp[:, :K].astype(np.int64).T
    assert np.array_equal(C[:, :N], ref)
    assert np.all(C[:, N:] == 0)
    del ctypes


# ------------------------------------------------------------- INT4 GEMM ----

def test_gemm_s4_all_value_pairs(oracle):
    vals = np.arange(-8, 8)
    A = np.zeros((16, 2), dtype=np.int8)
    B = np.zeros((16, 2), dtype=np.int8)
    A[:, 0] = vals
    B[:, 0] = vals
    C = oracle.gemm_s4(oracle.s4_pack(A), oracle.s4_pack(B), 2)
    assert np.array_equal(C, np.outer(vals, vals).astype(np.int32))


@pytest.mark.parametrize("M,N,K", [(1, 1, 2), (5, 3, 10), (33, 17, 64), (40, 70, 128)])
def test_gemm_s4_matches_numpy_int64(oracle, M, N, K):
    A = inputs.s8_in_range(M, K, -8, 7, 20 + M)
    B = inputs.s8_in_range(N, K, -8, 7, 21 + N)
    C = oracle.gemm_s4(oracle.s4_pack(A), oracle.s4_pack(B), K)
    assert np.array_equal(C.astype(np.int64), A.astype(np.int64) @ B.astype(np.int64).T)


def test_gemm_s4_closed_form_all_minus_eight(oracle):
    K = 4096
    P = np.full((2, K // 2), 0x88, dtype=np.uint8)
    assert np.all(oracle.gemm_s4(P, P, K) == 64 * K)


def test_gemm_s4_equals_gemm_s8_on_small_values(oracle):
    A = inputs.s8_in_range(12, 46, -8, 7, 30)
    B = inputs.s8_in_range(9, 46, -8, 7, 31)
    assert np.array_equal(oracle.gemm_s4(oracle.s4_pack(A), oracle.s4_pack(B), 46),
                          oracle.gemm_s8(A, B))


# ------------------------------------------------------------- FP16 GEMM ----

def test_gemm_f16_exact_on_integer_inputs(oracle):
    A = inputs.s8_in_range(11, 64, -16, 16, 40).astype(np.float16)
    B = inputs.s8_in_range(7, 64, -16, 16, 41).astype(np.float16)
    C = oracle.gemm_f16(A, B)
    ref = A.astype(np.int64) @ B.astype(np.int64).T
    assert np.array_equal(C, ref.astype(np.float64))


def test_gemm_f16_identity_gives_transpose(oracle):
    B = inputs.f16_normal(9, 32, 42)
    C = oracle.gemm_f16(np.eye(32, dtype=np.float16), B)
    assert np.array_equal(C, B.T.astype(np.float64))


def test_gemm_f16_matches_numpy_float64(oracle):
    A = inputs.f16_normal(37, 200, 43)
    B = inputs.f16_normal(29, 200, 44)
    C = oracle.gemm_f16(A, B)
    ref = A.astype(np.float64) @ B.astype(np.float64).T
    assert np.max(np.abs(C - ref)) <= 1e-12 * np.max(np.abs(ref))


# ---------------------------------------------------------------- W4A16 ----

def test_w4a16_unit_scale_integer_x_is_exact(oracle):
    M, N, K, g = 3, 10, 256, 128
    q = inputs.s8_in_range(N, K, -8, 7, 50)
    X = inputs.s8_in_range(M, K, -4, 4, 51)
    S = np.ones((N, K // g), dtype=np.float16)
    Y = oracle.w4a16(X.astype(np.float16), oracle.s4_pack(q), S, g)
    assert np.array_equal(Y, (X.astype(np.int64) @ q.astype(np.int64).T).astype(np.float64))


def test_w4a16_matches_dequantized_numpy_gemm(oracle):
    M, N, K, g = 5, 24, 512, 128
    q = inputs.s8_in_range(N, K, -8, 7, 52)
    X = inputs.f16_normal(M, K, 53)
    S = inputs.f16_uniform(N, K // g, 0.005, 0.02, 54)
    Y = oracle.w4a16(X, oracle.s4_pack(q), S, g)
    W = q.astype(np.float64) * np.repeat(S.astype(np.float64), g, axis=1)
    ref = X.astype(np.float64) @ W.T
    assert np.max(np.abs(Y - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_w4a16_group_indexing(oracle):
    # q = 1, X = 1: Y[n] = group * sum_g s[n, g]; distinct scales per (n, g)
    M, N, K, g = 1, 4, 512, 128
    q = np.ones((N, K), dtype=np.int8)
    S = (np.arange(N * (K // g)).reshape(N, K // g) + 1).astype(np.float16)
    Y = oracle.w4a16(np.ones((M, K), dtype=np.float16), oracle.s4_pack(q), S, g)
    assert np.array_equal(Y[0], g * S.astype(np.float64).sum(axis=1))


# ------------------------------------------------------- W4A4 quantizer ----

def _golden_quant_cases():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "w4a4_quantize.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tok = line.split()
            if tok[0] == "case":
                cur = {"name": tok[1], "entries": []}
            elif tok[0] == "scale_bits":
                cur["scale"] = int(tok[1], 16)
            elif tok[0] == "end":
                cases.append(cur)
            else:
                cur["entries"].append((int(tok[0]), float(tok[1]), int(tok[2])))
    return cases


@pytest.mark.parametrize("case", _golden_quant_cases(), ids=lambda c: c["name"])
def test_w4a4_quantize_golden(oracle, case):
    X = np.zeros((1, 64), dtype=np.float32)
    for i, x, _ in case["entries"]:
        X[0, i] = np.float32(x)
    Q, S = oracle.w4a4_quantize(X, 64)
    assert S[0, 0] == case["scale"]
    q = oracle.s4_unpack(Q, 64)[0]
    expect = np.zeros(64, dtype=np.int8)
    for i, _, qi in case["entries"]:
        expect[i] = qi
    assert np.array_equal(q, expect)


def test_w4a4_quantize_invariants(oracle):
    M, K, blk = 16, 512, 64
    X = inputs.f32_normal(M, K, 60)
    Q, S = oracle.w4a4_quantize(X, blk)
    q = oracle.s4_unpack(Q, K).astype(np.float64)
    s = np.repeat(S.view(np.float16).astype(np.float64), blk, axis=1)
    # absmax maps to +-7 in every (non-zero) block
    assert np.all(np.abs(q).reshape(M, K // blk, blk).max(axis=2) == 7)
    # rounding error at most half a step
    assert np.all(np.abs(X.astype(np.float64) - q * s) <= s / 2 + 1e-12)
    # the scale is the rounded absmax / 7, per row and block (not transposed)
    a = np.abs(X).reshape(M, K // blk, blk).max(axis=2)
    assert np.array_equal(S.view(np.float16), (a / np.float32(7)).astype(np.float16))


def test_w4a4_quantize_is_idempotent(oracle):
    X = inputs.f32_normal(8, 256, 61)
    Q, S = oracle.w4a4_quantize(X, 64)
    q = oracle.s4_unpack(Q, 256).astype(np.float32)
    Xd = q * np.repeat(S.view(np.float16).astype(np.float32), 64, axis=1)
    Q2, S2 = oracle.w4a4_quantize(Xd.astype(np.float32), 64)
    assert np.array_equal(Q2, Q) and np.array_equal(S2, S)


def test_lowrank_xu_matches_numpy(oracle):
    X = inputs.f32_normal(6, 300, 62)
    U = inputs.f16_normal(300, 32, 63, sigma=0.02)
    XU = oracle.lowrank_xu(X, U)
    ref = X.astype(np.float64) @ U.astype(np.float64)
    assert np.max(np.abs(XU - ref)) <= 1e-12 * np.max(np.abs(ref))


# ------------------------------------------------------------ W4A4 GEMM ----

def _w4a4_operands(M, N, K, blk, seed, pow2_scales=False):
    qx = inputs.s8_in_range(M, K, -8, 7, seed)
    qw = inputs.s8_in_range(N, K, -8, 7, seed + 1)
    if pow2_scales:
        ex = inputs.s8_in_range(M, K // blk, -6, 2, seed + 2).astype(np.float64)
        ew = inputs.s8_in_range(N, K // blk, -6, 2, seed + 3).astype(np.float64)
        sx, sw = (2.0 ** ex).astype(np.float16), (2.0 ** ew).astype(np.float16)
    else:
        sx = inputs.f16_uniform(M, K // blk, 0.01, 0.5, seed + 2)
        sw = inputs.f16_uniform(N, K // blk, 0.01, 0.5, seed + 3)
    return qx, qw, sx, sw


def _blockwise_numpy(qx, qw, sx, sw, blk):
    M, K = qx.shape
    out = np.zeros((M, qw.shape[0]))
    for j in range(K // blk):
        sl = slice(j * blk, (j + 1) * blk)
        dots = qx[:, sl].astype(np.int64) @ qw[:, sl].astype(np.int64).T
        out += np.outer(sx[:, j].astype(np.float64), sw[:, j].astype(np.float64)) * dots
    return out


def test_w4a4_gemm_no_lowrank_equals_blockwise_scaled_integer_gemm(oracle):
    M, N, K, blk = 9, 11, 256, 64
    qx, qw, sx, sw = _w4a4_operands(M, N, K, blk, 70)
    Y = oracle.w4a4_gemm(oracle.s4_pack(qx), sx, oracle.s4_pack(qw), sw, blk, K)
    ref = _blockwise_numpy(qx, qw, sx, sw, blk)
    assert np.max(np.abs(Y - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_w4a4_gemm_power_of_two_scales_exact(oracle):
    M, N, K, blk = 7, 5, 192, 64
    qx, qw, sx, sw = _w4a4_operands(M, N, K, blk, 80, pow2_scales=True)
    Y = oracle.w4a4_gemm(oracle.s4_pack(qx), sx, oracle.s4_pack(qw), sw, blk, K)
    assert np.array_equal(Y, _blockwise_numpy(qx, qw, sx, sw, blk))


def test_w4a4_gemm_unit_scales_equals_int4_gemm(oracle):
    M, N, K, blk = 6, 8, 128, 64
    qx, qw, _, _ = _w4a4_operands(M, N, K, blk, 90)
    one_x = np.ones((M, K // blk), dtype=np.float16)
    one_w = np.ones((N, K // blk), dtype=np.float16)
    px, pw = oracle.s4_pack(qx), oracle.s4_pack(qw)
    Y = oracle.w4a4_gemm(px, one_x, pw, one_w, blk, K)
    assert np.array_equal(Y, oracle.gemm_s4(px, pw, K).astype(np.float64))


def test_w4a4_gemm_lowrank_and_bias(oracle):
    M, N, K, blk, R = 5, 12, 128, 64, 32
    qx, qw, sx, sw = _w4a4_operands(M, N, K, blk, 100)
    XU = inputs.f32_normal(M, R, 104).astype(np.float64)
    V = inputs.f16_normal(R, N, 105, sigma=0.02)
    b = inputs.f16_normal(1, N, 106, sigma=0.1)[0]
    Y = oracle.w4a4_gemm(oracle.s4_pack(qx), sx, oracle.s4_pack(qw), sw, blk, K,
                         XU=XU, V=V, bias=b)
    ref = (_blockwise_numpy(qx, qw, sx, sw, blk) + XU @ V.astype(np.float64)
           + b.astype(np.float64)[None, :])
    assert np.max(np.abs(Y - ref)) <= 1e-12 * np.max(np.abs(ref))


# The column-wise affine calibration of the W4A4 page (sections 1 and 5.2),
# read as t -> alpha[n] * t + b[n] on every output column, where t is the
# block-scaled product plus the low-rank term.

def test_w4a4_gemm_unit_alpha_is_the_printed_formula(oracle):
    M, N, K, blk, R = 4, 9, 128, 64, 32
    qx, qw, sx, sw = _w4a4_operands(M, N, K, blk, 110)
    XU = inputs.f32_normal(M, R, 114).astype(np.float64)
    V = inputs.f16_normal(R, N, 115, sigma=0.02)
    b = inputs.f16_normal(1, N, 116, sigma=0.1)[0]
    args = (oracle.s4_pack(qx), sx, oracle.s4_pack(qw), sw, blk, K)
    Y0 = oracle.w4a4_gemm(*args, XU=XU, V=V, bias=b)
    Y1 = oracle.w4a4_gemm(*args, XU=XU, V=V, bias=b, alpha=np.ones(N, dtype=np.float16))
    assert np.array_equal(Y0, Y1)


def test_w4a4_gemm_alpha_scales_product_and_lowrank_not_bias(oracle):
    M, N, K, blk, R = 5, 12, 192, 64, 32
    qx, qw, sx, sw = _w4a4_operands(M, N, K, blk, 120, pow2_scales=True)
    # alpha and every other operand exact in binary: the result is exact
    alpha = (2.0 ** inputs.s8_in_range(1, N, -3, 3, 121)[0].astype(np.float64)).astype(np.float16)
    XU = inputs.s8_in_range(M, R, -4, 4, 124).astype(np.float64)
    V = (inputs.s8_in_range(R, N, -4, 4, 125).astype(np.float64) / 8).astype(np.float16)
    b = (inputs.s8_in_range(1, N, -16, 16, 126)[0].astype(np.float64) / 4).astype(np.float16)
    Y = oracle.w4a4_gemm(oracle.s4_pack(qx), sx, oracle.s4_pack(qw), sw, blk, K,
                         XU=XU, V=V, bias=b, alpha=alpha)
    a = alpha.astype(np.float64)[None, :]
    t = _blockwise_numpy(qx, qw, sx, sw, blk) + XU @ V.astype(np.float64)
    assert np.array_equal(Y, a * t + b.astype(np.float64)[None, :])
    # zero codes: only the low-rank term, scaled by alpha, plus the bias
    z = np.zeros_like(qx)
    Yz = oracle.w4a4_gemm(oracle.s4_pack(z), sx, oracle.s4_pack(qw), sw, blk, K,
                          XU=XU, V=V, bias=b, alpha=alpha)
    assert np.array_equal(Yz, a * (XU @ V.astype(np.float64)) + b.astype(np.float64)[None, :])
    # no low-rank term, no bias: alpha times the block-scaled product
    Yp = oracle.w4a4_gemm(oracle.s4_pack(qx), sx, oracle.s4_pack(qw), sw, blk, K, alpha=alpha)
    assert np.array_equal(Yp, a * _blockwise_numpy(qx, qw, sx, sw, blk))


def test_w4a4_gemm_alpha_matches_numpy(oracle):
    M, N, K, blk, R = 6, 10, 256, 64, 32
    qx, qw, sx, sw = _w4a4_operands(M, N, K, blk, 130)
    alpha = inputs.f16_uniform(1, N, 0.5, 2.0, 131)[0]
    XU = inputs.f32_normal(M, R, 134).astype(np.float64)
    V = inputs.f16_normal(R, N, 135, sigma=0.02)
    b = inputs.f16_normal(1, N, 136, sigma=0.1)[0]
    Y = oracle.w4a4_gemm(oracle.s4_pack(qx), sx, oracle.s4_pack(qw), sw, blk, K,
                         XU=XU, V=V, bias=b, alpha=alpha)
    ref = (alpha.astype(np.float64)[None, :]
           * (_blockwise_numpy(qx, qw, sx, sw, blk) + XU @ V.astype(np.float64))
           + b.astype(np.float64)[None, :])
    assert np.max(np.abs(Y - ref)) <= 1e-12 * np.max(np.abs(ref))
