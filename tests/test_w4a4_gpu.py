"""GPU parity of w4a4_quantize (bit-exact) and w4a4_gemm (fp16 tolerance)."""
import os

import numpy as np
import pytest

from bit_quantized_tensor_gb300 import inputs
from tests._util import assert_fp16_close

pytestmark = pytest.mark.gpu

BLOCK, RANK = 64, 32
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def dev():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import bit_quantized_tensor_gb300 as qg
    qg.lib()
    return torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _no_device_timeouts(dev):
    import bit_quantized_tensor_gb300 as qg
    yield
    assert qg.device_status() == qg.QG_OK


def _t(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def _quant(dev, X, U=None):
    import bit_quantized_tensor_gb300 as qg
    q, s, xu = qg.w4a4_quantize(_t(X, dev), None if U is None else _t(U.T, dev), BLOCK)
    return (q.cpu().numpy(), s.cpu().numpy().view(np.uint16),
            None if xu is None else xu.cpu().numpy())


# ------------------------------------------------------------- quantizer

@pytest.mark.parametrize("M,K", [(1, 64), (17, 128), (100, 512), (16, 8192), (33, 1088)])
def test_quantize_bit_exact(dev, oracle, M, K):
    X = inputs.f32_normal(M, K, 1004 + M)
    q, s, _ = _quant(dev, X)
    q_ref, s_ref = oracle.w4a4_quantize(X, BLOCK)
    assert np.array_equal(s, s_ref)
    assert np.array_equal(q, q_ref)


def test_quantize_golden_edge_cases(dev, oracle):
    # the hand-derived blocks (ties to even, fp16-subnormal scale with clamping,
    # all-zero block), one per row
    from tests.test_oracle import _golden_quant_cases
    cases = _golden_quant_cases()
    X = np.zeros((len(cases), BLOCK), dtype=np.float32)
    for r, c in enumerate(cases):
        for i, x, _ in c["entries"]:
            X[r, i] = np.float32(x)
    q, s, _ = _quant(dev, X)
    for r, c in enumerate(cases):
        assert s[r, 0] == c["scale"], c["name"]
        vals = oracle.s4_unpack(q[r:r + 1], BLOCK)[0]
        for i, _, qi in c["entries"]:
            assert vals[i] == qi, (c["name"], i)


def _near_tie_blocks(M, K, seed):
    """Blocks whose values sit a few ulps either side of (k + 1/2) * s.

    Each block's first value is 7 * s0 for an fp16 value s0, so the block
    scale is exactly s0; every other value is (k + 1/2) * s0, exact in fp32,
    moved by -6..6 ulps.  x / s then lands within a few ulps of a rounding
    tie, on either side of it or on it.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    nb = K // BLOCK
    s0 = rng.uniform(-14.0, 3.0, size=(M, nb))
    s0 = (2.0 ** s0).astype(np.float16).astype(np.float32)
    s0[:, 0] = np.float32(np.float16(2.0 ** -23))       # fp16-subnormal scales
    s0[:, 1] = np.float32(np.float16(0.3))              # 1 / s inexact
    h = rng.integers(-7, 7, size=(M, K)).astype(np.float32) + np.float32(0.5)
    base = (h * np.repeat(s0, BLOCK, axis=1)).astype(np.float32)
    d = rng.integers(-6, 7, size=(M, K)).astype(np.int32)
    mag = (np.abs(base).view(np.int32) + d).view(np.float32)
    X = np.where(base < 0, -mag, mag).astype(np.float32)
    X[:, ::BLOCK] = 7.0 * s0
    return X


def test_quantize_near_ties_bit_exact(dev, oracle):
    M, K = 48, 2048
    X = _near_tie_blocks(M, K, 91)
    q, s, _ = _quant(dev, X)
    q_ref, s_ref = oracle.w4a4_quantize(X, BLOCK)
    assert np.array_equal(s, s_ref)
    assert np.array_equal(q, q_ref)


def test_quantize_scaled_ranges_bit_exact(dev, oracle):
    # blocks spanning many magnitudes, including fp16-subnormal and overflowing scales
    M, K = 64, 1024
    X = inputs.f32_normal(M, K, 77)
    mags = (10.0 ** inputs.s8_in_range(M, K // BLOCK, -9, 5, 78)).astype(np.float32)
    X = X * np.repeat(mags, BLOCK, axis=1)
    q, s, _ = _quant(dev, X)
    q_ref, s_ref = oracle.w4a4_quantize(X, BLOCK)
    assert np.array_equal(s, s_ref)
    assert np.array_equal(q, q_ref)


@pytest.mark.parametrize("M,K", [(5, 64), (40, 1024), (300, 2048)])
def test_quantize_lowrank_projection(dev, oracle, M, K):
    X = inputs.f32_normal(M, K, 1104 + M)
    U = inputs.f16_normal(K, RANK, 3104, sigma=0.02)
    q, s, xu = _quant(dev, X, U)
    q_ref, s_ref = oracle.w4a4_quantize(X, BLOCK)
    assert np.array_equal(q, q_ref) and np.array_equal(s, s_ref)
    assert_fp16_close(xu, oracle.lowrank_xu(X, U), f"XU {M}x{K}")


def test_quantize_full_size(dev, oracle):
    # the W4A4 workload's activations: 4096 x 8192 fp32, every code and scale
    X = inputs.f32_normal(4096, 8192, 1004)
    U = inputs.f16_normal(8192, RANK, 3004, sigma=0.02)
    q, s, xu = _quant(dev, X, U)
    q_ref, s_ref = oracle.w4a4_quantize(X, BLOCK)
    assert np.array_equal(s, s_ref)
    assert np.array_equal(q, q_ref)
    rows = inputs.sample_rows(4096, 64, 5004)
    assert_fp16_close(xu[rows], oracle.lowrank_xu(X[rows], U), "XU full size sampled")


# ------------------------------------------------------------------ GEMM

def _gemm_case(M, N, K, seed, rank=RANK, with_bias=True):
    X = inputs.f32_normal(M, K, 1000 + seed)
    W = inputs.f32_normal(N, K, 2000 + seed)
    U = inputs.f16_normal(K, RANK, 3000 + seed, sigma=0.02)
    V = inputs.f16_normal(RANK, N, 3100 + seed, sigma=0.02)
    b = inputs.f16_normal(1, N, 3200 + seed, sigma=0.1)[0] if with_bias else None
    return X, W, U, V, b


@pytest.fixture
def gemm_path():
    import bit_quantized_tensor_gb300 as qg
    def set_path(p):
        assert qg.lib().qg_set_gemm_path(p) == 0
    yield set_path
    qg.lib().qg_set_gemm_path(0)


GEMM_SHAPES = [(1, 8, 64, 32, True), (100, 300, 256, 32, True), (129, 257, 576, 32, False),
               (64, 512, 1024, 0, True), (256, 256, 4096, 0, False), (300, 136, 192, 32, True),
               (520, 392, 1088, 32, True)]


@pytest.mark.parametrize("path", [0, 1, 2])
@pytest.mark.parametrize("M,N,K,rank,bias", GEMM_SHAPES)
def test_gemm_matches_oracle(dev, oracle, gemm_path, path, M, N, K, rank, bias):
    import bit_quantized_tensor_gb300 as qg
    gemm_path(path)
    X, W, U, V, b = _gemm_case(M, N, K, 7, rank, bias)
    qx, sx = oracle.w4a4_quantize(X, BLOCK)
    qw, sw = oracle.w4a4_quantize(W, BLOCK)
    xu16 = oracle.lowrank_xu(X, U).astype(np.float16) if rank else None
    Y = qg.w4a4_gemm(_t(qx, dev), _t(sx.view(np.float16), dev), _t(qw, dev),
                     _t(sw.view(np.float16), dev), K,
                     XU=_t(xu16, dev) if rank else None, Vt=_t(V.T, dev) if rank else None,
                     bias=_t(b, dev) if bias else None).cpu().numpy()
    ref = oracle.w4a4_gemm(qx, sx, qw, sw, BLOCK, K,
                           XU=xu16.astype(np.float64) if rank else None,
                           V=V if rank else None, bias=b if bias else None)
    assert_fp16_close(Y, ref, f"w4a4 {M}x{N}x{K} r={rank}")


@pytest.mark.parametrize("path", [1, 2])
def test_gemm_unit_scales_equal_int4_gemm(dev, oracle, gemm_path, path):
    # sX = sW = 1 and no low-rank term: Y is the INT4 GEMM rounded to fp16
    # (exact while |Y| <= 2048)
    import bit_quantized_tensor_gb300 as qg
    gemm_path(path)
    M, N, K = 96, 160, 64
    qx = inputs.s4_packed_uniform(M, K, 21)
    qw = inputs.s4_packed_uniform(N, K, 22)
    one_x = np.ones((M, K // BLOCK), dtype=np.float16)
    one_w = np.ones((N, K // BLOCK), dtype=np.float16)
    Y = qg.w4a4_gemm(_t(qx, dev), _t(one_x, dev), _t(qw, dev), _t(one_w, dev), K).cpu().numpy()
    assert np.array_equal(Y.astype(np.float64), oracle.gemm_s4(qx, qw, K).astype(np.float64))


AFFINE_SHAPES = [(1, 8, 64, 32, True), (100, 300, 256, 32, True), (300, 136, 192, 0, False),
                 (520, 392, 1088, 32, True)]


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("M,N,K,rank,bias", AFFINE_SHAPES)
def test_gemm_affine_matches_oracle(dev, oracle, gemm_path, path, M, N, K, rank, bias):
    """Column-wise affine calibration: Y = alpha (.) (scaled product + L(X)) + b."""
    import bit_quantized_tensor_gb300 as qg
    gemm_path(path)
    X, W, U, V, b = _gemm_case(M, N, K, 11, rank, bias)
    alpha = inputs.f16_uniform(1, N, 0.25, 4.0, 3300 + M)[0]
    qx, sx = oracle.w4a4_quantize(X, BLOCK)
    qw, sw = oracle.w4a4_quantize(W, BLOCK)
    xu16 = oracle.lowrank_xu(X, U).astype(np.float16) if rank else None
    Y = qg.w4a4_gemm(_t(qx, dev), _t(sx.view(np.float16), dev), _t(qw, dev),
                     _t(sw.view(np.float16), dev), K,
                     XU=_t(xu16, dev) if rank else None, Vt=_t(V.T, dev) if rank else None,
                     bias=_t(b, dev) if bias else None, alpha=_t(alpha, dev)).cpu().numpy()
    ref = oracle.w4a4_gemm(qx, sx, qw, sw, BLOCK, K,
                           XU=xu16.astype(np.float64) if rank else None,
                           V=V if rank else None, bias=b if bias else None, alpha=alpha)
    assert_fp16_close(Y, ref, f"w4a4 affine {M}x{N}x{K} r={rank}")


def test_gemm_affine_unit_alpha_equals_plain_call(dev, oracle):
    """alpha = 1 gives bit for bit the plain w4a4_gemm result."""
    import bit_quantized_tensor_gb300 as qg
    M, N, K = 260, 384, 512
    X, W, U, V, b = _gemm_case(M, N, K, 12)
    tX, tW = _t(X, dev), _t(W, dev)
    qx, sx, xu = qg.w4a4_quantize(tX, _t(U.T, dev), BLOCK)
    qw, sw, _ = qg.w4a4_quantize(tW, None, BLOCK)
    Vt, tb = _t(V.T, dev), _t(b, dev)
    Y0 = qg.w4a4_gemm(qx, sx, qw, sw, K, XU=xu, Vt=Vt, bias=tb).cpu().numpy()
    one = _t(np.ones(N, dtype=np.float16), dev)
    Y1 = qg.w4a4_gemm(qx, sx, qw, sw, K, XU=xu, Vt=Vt, bias=tb, alpha=one).cpu().numpy()
    assert np.array_equal(Y0.view(np.uint16), Y1.view(np.uint16))


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("M,N,K,rank,bias,affine", [(100, 300, 256, 32, True, False),
                                                    (520, 392, 1088, 32, True, True),
                                                    (129, 257, 576, 0, False, False)])
def test_prepacked_weights_give_the_same_bits(dev, oracle, gemm_path, path, M, N, K, rank, bias, affine):
    """w4a4_prepack_weights + w4a4_gemm_prepacked against w4a4_gemm (or
    w4a4_gemm_affine) on the same inputs: the same bits, and the oracle."""
    import bit_quantized_tensor_gb300 as qg
    gemm_path(path)
    X, W, U, V, b = _gemm_case(M, N, K, 13, rank, bias)
    alpha = inputs.f16_uniform(1, N, 0.5, 2.0, 3500 + M)[0] if affine else None
    qx, sx, xu = qg.w4a4_quantize(_t(X, dev), _t(U.T, dev) if rank else None, BLOCK)
    qw, sw, _ = qg.w4a4_quantize(_t(W, dev), None, BLOCK)
    ta = _t(alpha, dev) if affine else None
    kw = dict(XU=xu if rank else None, Vt=_t(V.T, dev) if rank else None, bias=_t(b, dev) if bias else None)
    Y0 = qg.w4a4_gemm(qx, sx, qw, sw, K, alpha=ta, **kw).cpu().numpy()
    packed = qg.w4a4_prepack_weights(qw, sw, K, alpha=ta)
    Y1 = qg.w4a4_gemm_prepacked(qx, sx, packed, N, K, **kw).cpu().numpy()
    Y2 = qg.w4a4_gemm_prepacked(qx, sx, packed, N, K, **kw).cpu().numpy()  # the buffer is reusable
    assert np.array_equal(Y0.view(np.uint16), Y1.view(np.uint16))
    assert np.array_equal(Y1.view(np.uint16), Y2.view(np.uint16))
    qx_r, sx_r = oracle.w4a4_quantize(X, BLOCK)
    qw_r, sw_r = oracle.w4a4_quantize(W, BLOCK)
    ref = oracle.w4a4_gemm(qx_r, sx_r, qw_r, sw_r, BLOCK, K,
                           XU=xu.cpu().numpy().astype(np.float64) if rank else None,
                           V=V if rank else None, bias=b if bias else None, alpha=alpha)
    assert_fp16_close(Y1, ref, f"w4a4 prepacked {M}x{N}x{K}")


def test_end_to_end_full_size_sampled(dev, oracle):
    """The W4A4 workload (M=4096, N=K=8192, rank 32): GPU quantizer + GPU GEMM
    against the oracle's quantize -> X.U -> block-scaled GEMM on sampled rows."""
    import bit_quantized_tensor_gb300 as qg
    M, N, K = 4096, 8192, 8192
    X, W, U, V, b = _gemm_case(M, N, K, 4)
    tX, tW = _t(X, dev), _t(W, dev)
    qx, sx, xu = qg.w4a4_quantize(tX, _t(U.T, dev), BLOCK)
    qw, sw, _ = qg.w4a4_quantize(tW, None, BLOCK)
    Y = qg.w4a4_gemm(qx, sx, qw, sw, K, XU=xu, Vt=_t(V.T, dev), bias=_t(b, dev)).cpu().numpy()
    rows = inputs.sample_rows(M, 24, 5104)
    qx_r, sx_r = oracle.w4a4_quantize(X[rows], BLOCK)
    qw_r, sw_r = oracle.w4a4_quantize(W, BLOCK)
    ref = oracle.w4a4_gemm(qx_r, sx_r, qw_r, sw_r, BLOCK, K, XU=oracle.lowrank_xu(X[rows], U),
                           V=V, bias=b)
    assert_fp16_close(Y[rows], ref, "w4a4 end to end")
