"""GPU parity of gemm_f16, qgemm_s8 and qgemm_s4 against the CPU oracle.

Integer results must be bit-exact; fp16 results must meet the stated
tolerance.  Large sizes compare sampled rows with the oracle and the whole
product with Freivalds' randomized identity.
"""
import numpy as np
import pytest

from bit_quantized_tensor_gb300 import inputs
from tests._util import assert_fp16_close, first_mismatch, freivalds_int

pytestmark = pytest.mark.gpu


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


# ------------------------------------------------------------------ gemm_f16

@pytest.mark.parametrize("M,N,K", [(1, 1, 8), (100, 300, 136), (128, 256, 64), (129, 257, 72),
                                   (384, 768, 1024), (256, 512, 200)])
def test_gemm_f16_shapes(dev, oracle, M, N, K):
    import bit_quantized_tensor_gb300 as qg
    A = inputs.f16_normal(M, K, 1000 + M)
    B = inputs.f16_normal(N, K, 2000 + N)
    C = qg.gemm_f16(_t(A, dev), _t(B, dev)).cpu().numpy()
    assert_fp16_close(C, oracle.gemm_f16(A, B), f"gemm_f16 {M}x{N}x{K}")


@pytest.mark.parametrize("n", [512, 1024, 2048])
def test_gemm_f16_sweep_full(dev, oracle, n):
    import bit_quantized_tensor_gb300 as qg
    A = inputs.f16_normal(n, n, 1002)
    B = inputs.f16_normal(n, n, 2002)
    C = qg.gemm_f16(_t(A, dev), _t(B, dev)).cpu().numpy()
    assert_fp16_close(C, oracle.gemm_f16(A, B), f"gemm_f16 {n}")


@pytest.mark.parametrize("n", [4096, 8192])
def test_gemm_f16_sweep_sampled(dev, oracle, n):
    import bit_quantized_tensor_gb300 as qg
    A = inputs.f16_normal(n, n, 1002)
    B = inputs.f16_normal(n, n, 2002)
    C = qg.gemm_f16(_t(A, dev), _t(B, dev)).cpu().numpy()
    rows = inputs.sample_rows(n, 48, 4000 + n)
    assert_fp16_close(C[rows], oracle.gemm_f16(A[rows], B), f"gemm_f16 {n} sampled")


def test_gemm_f16_identity(dev):
    import bit_quantized_tensor_gb300 as qg
    B = inputs.f16_normal(200, 64, 5)
    C = qg.gemm_f16(_t(np.eye(64, dtype=np.float16), dev), _t(B, dev)).cpu().numpy()
    assert np.array_equal(C, B.T)


# ------------------------------------------------------------------ qgemm_s8

def _s8(dev, A, B):
    import bit_quantized_tensor_gb300 as qg
    return qg.qgemm_s8(_t(A, dev), _t(B, dev)).cpu().numpy()


def test_qgemm_s8_int8_512(dev, oracle):
    A = inputs.s8_uniform(512, 512, 1000)
    B = inputs.s8_uniform(512, 512, 2000)
    C = _s8(dev, A, B)
    ref = oracle.gemm_s8(A, B)
    assert np.array_equal(C, ref), first_mismatch(C, ref)


@pytest.mark.parametrize("M,N,K", [(1, 1, 16), (77, 300, 48), (130, 260, 1040), (200, 513, 2064),
                                   (128, 256, 1024), (300, 129, 3072)])
def test_qgemm_s8_shapes(dev, oracle, M, N, K):
    A = inputs.s8_uniform(M, K, 1100 + M)
    B = inputs.s8_uniform(N, K, 2100 + N)
    C = _s8(dev, A, B)
    ref = oracle.gemm_s8(A, B)
    assert np.array_equal(C, ref), first_mismatch(C, ref)


@pytest.mark.parametrize("K", [1024, 4096, 8192])
def test_qgemm_s8_extremes(dev, K):
    # -128 * -128 summed over a 1024 chunk is exactly 2^24: the largest
    # partial sum the fp32 accumulator must carry exactly.
    A = np.full((256, K), -128, dtype=np.int8)
    B = np.full((256, K), -128, dtype=np.int8)
    B[128:] = 127
    C = _s8(dev, A, B)
    assert np.all(C[:, :128] == 16384 * K)
    assert np.all(C[:, 128:] == -16256 * K)


@pytest.mark.parametrize("chunk", [1, 5, 16])
def test_qgemm_s8_chunk_lengths(dev, oracle, chunk):
    import bit_quantized_tensor_gb300 as qg
    A = inputs.s8_uniform(192, 2112, 1200)
    B = inputs.s8_uniform(320, 2112, 2200)
    assert qg.lib().qg_set_s8_chunk(chunk) == 0
    try:
        C = _s8(dev, A, B)
    finally:
        qg.lib().qg_set_s8_chunk(16)
    ref = oracle.gemm_s8(A, B)
    assert np.array_equal(C, ref), first_mismatch(C, ref)


@pytest.mark.parametrize("n", [1024, 2048])
def test_qgemm_s8_sweep_full(dev, oracle, n):
    A = inputs.s8_uniform(n, n, 1002)
    B = inputs.s8_uniform(n, n, 2002)
    C = _s8(dev, A, B)
    ref = oracle.gemm_s8(A, B)
    assert np.array_equal(C, ref), first_mismatch(C, ref)


@pytest.mark.parametrize("n", [4096, 8192])
def test_qgemm_s8_sweep_large(dev, oracle, n):
    A = inputs.s8_uniform(n, n, 1002)
    B = inputs.s8_uniform(n, n, 2002)
    C = _s8(dev, A, B)
    rows = inputs.sample_rows(n, 64, 4100 + n)
    ref = oracle.gemm_s8(A[rows], B)
    assert np.array_equal(C[rows], ref), first_mismatch(C[rows], ref)
    freivalds_int(A, B, C)


# ------------------------------------------------------------------ qgemm_s4

def _s4(dev, A, B, K):
    import bit_quantized_tensor_gb300 as qg
    return qg.qgemm_s4(_t(A, dev), _t(B, dev), K).cpu().numpy()


def test_qgemm_s4_int4_2048(dev, oracle):
    A = inputs.s4_packed_uniform(2048, 2048, 1001)
    B = inputs.s4_packed_uniform(2048, 2048, 2001)
    C = _s4(dev, A, B, 2048)
    ref = oracle.gemm_s4(A, B, 2048)
    assert np.array_equal(C, ref), first_mismatch(C, ref)


@pytest.mark.parametrize("M,N,K", [(1, 1, 32), (77, 300, 96), (130, 260, 1056), (200, 513, 4160),
                                   (128, 256, 128)])
def test_qgemm_s4_shapes(dev, oracle, M, N, K):
    A = inputs.s4_packed_uniform(M, K, 1300 + M)
    B = inputs.s4_packed_uniform(N, K, 2300 + N)
    C = _s4(dev, A, B, K)
    ref = oracle.gemm_s4(A, B, K)
    assert np.array_equal(C, ref), first_mismatch(C, ref)


@pytest.mark.parametrize("K", [1024, 8192, 32768])
def test_qgemm_s4_extremes(dev, K):
    A = np.full((128, K // 2), 0x88, dtype=np.uint8)       # all -8
    B = np.full((256, K // 2), 0x88, dtype=np.uint8)
    B[128:] = 0x77                                          # all 7
    C = _s4(dev, A, B, K)
    assert np.all(C[:, :128] == 64 * K)
    assert np.all(C[:, 128:] == -56 * K)


def test_qgemm_s4_matches_s8_on_same_values(dev, oracle):
    vals_a = inputs.s8_in_range(160, 512, -8, 7, 1400)
    vals_b = inputs.s8_in_range(300, 512, -8, 7, 2400)
    C4 = _s4(dev, oracle.s4_pack(vals_a), oracle.s4_pack(vals_b), 512)
    C8 = _s8(dev, vals_a, vals_b)
    assert np.array_equal(C4, C8)
    assert np.array_equal(C4, oracle.gemm_s8(vals_a, vals_b))


@pytest.mark.parametrize("n", [512, 1024])
def test_qgemm_s4_sweep_full(dev, oracle, n):
    A = inputs.s4_packed_uniform(n, n, 1002)
    B = inputs.s4_packed_uniform(n, n, 2002)
    C = _s4(dev, A, B, n)
    ref = oracle.gemm_s4(A, B, n)
    assert np.array_equal(C, ref), first_mismatch(C, ref)


@pytest.mark.parametrize("n", [4096, 8192])
def test_qgemm_s4_sweep_large(dev, oracle, n):
    A = inputs.s4_packed_uniform(n, n, 1002)
    B = inputs.s4_packed_uniform(n, n, 2002)
    C = _s4(dev, A, B, n)
    rows = inputs.sample_rows(n, 64, 4200 + n)
    ref = oracle.gemm_s4(A[rows], B, n)
    assert np.array_equal(C[rows], ref), first_mismatch(C[rows], ref)
    freivalds_int(oracle.s4_unpack(A, n), oracle.s4_unpack(B, n), C)


# ------------------------------------------- both tensor-core kernel paths

@pytest.fixture
def gemm_path():
    import bit_quantized_tensor_gb300 as qg
    def set_path(p):
        assert qg.lib().qg_set_gemm_path(p) == 0
    yield set_path
    qg.lib().qg_set_gemm_path(0)


PATH_SHAPES = [(1, 1, 32), (300, 300, 1056), (257, 520, 96), (520, 260, 2112), (256, 256, 64),
               (640, 1000, 512)]


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("M,N,K", PATH_SHAPES)
def test_paths_qgemm_s8(dev, oracle, gemm_path, path, M, N, K):
    gemm_path(path)
    A = inputs.s8_uniform(M, K, 1500 + M)
    B = inputs.s8_uniform(N, K, 2500 + N)
    C = _s8(dev, A, B)
    ref = oracle.gemm_s8(A, B)
    assert np.array_equal(C, ref), first_mismatch(C, ref)


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("M,N,K", PATH_SHAPES)
def test_paths_qgemm_s4(dev, oracle, gemm_path, path, M, N, K):
    gemm_path(path)
    A = inputs.s4_packed_uniform(M, K, 1600 + M)
    B = inputs.s4_packed_uniform(N, K, 2600 + N)
    C = _s4(dev, A, B, K)
    ref = oracle.gemm_s4(A, B, K)
    assert np.array_equal(C, ref), first_mismatch(C, ref)


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("M,N,K", PATH_SHAPES)
def test_paths_gemm_f16(dev, oracle, gemm_path, path, M, N, K):
    import bit_quantized_tensor_gb300 as qg
    gemm_path(path)
    A = inputs.f16_normal(M, K, 1700 + M)
    B = inputs.f16_normal(N, K, 2700 + N)
    C = qg.gemm_f16(_t(A, dev), _t(B, dev)).cpu().numpy()
    assert_fp16_close(C, oracle.gemm_f16(A, B), f"gemm_f16 path {path} {M}x{N}x{K}")


# ------------------------------------------------- L2 cache-policy modes

@pytest.fixture
def l2_policy():
    import bit_quantized_tensor_gb300 as qg
    def set_mode(m):
        assert qg.lib().qg_set_l2_policy(m) == 0
    yield set_mode
    qg.lib().qg_set_l2_policy(0)


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("path", [1, 2])
def test_l2_policy_modes_same_results(dev, oracle, gemm_path, l2_policy, mode, path):
    """The cache hints change only where lines live in L2: the integer GEMMs
    stay bit-exact and the fp16 GEMM gives the same bits as mode 0."""
    import bit_quantized_tensor_gb300 as qg
    gemm_path(path)
    M, N, K = 520, 1000, 1056
    A = inputs.s8_uniform(M, K, 1800)
    B = inputs.s8_uniform(N, K, 2800)
    A4 = inputs.s4_packed_uniform(M, K, 1801)
    B4 = inputs.s4_packed_uniform(N, K, 2801)
    Af = inputs.f16_normal(M, K, 1802)
    Bf = inputs.f16_normal(N, K, 2802)
    l2_policy(0)
    f0 = qg.gemm_f16(_t(Af, dev), _t(Bf, dev)).cpu().numpy()
    l2_policy(mode)
    C8 = _s8(dev, A, B)
    ref = oracle.gemm_s8(A, B)
    assert np.array_equal(C8, ref), first_mismatch(C8, ref)
    C4 = _s4(dev, A4, B4, K)
    ref4 = oracle.gemm_s4(A4, B4, K)
    assert np.array_equal(C4, ref4), first_mismatch(C4, ref4)
    f1 = qg.gemm_f16(_t(Af, dev), _t(Bf, dev)).cpu().numpy()
    assert np.array_equal(f0.view(np.uint16), f1.view(np.uint16))


# ------------------------------------- qgemm_s4: in-kernel conversion vs pre-pass

@pytest.fixture
def s4_path():
    import bit_quantized_tensor_gb300 as qg
    def set_path(p):
        assert qg.lib().qg_set_s4_path(p) == 0
    yield set_path
    qg.lib().qg_set_s4_path(0)


@pytest.mark.parametrize("path", [0, 1])
@pytest.mark.parametrize("K", [1024, 65536])
def test_qgemm_s4_extremes_on_pairs(dev, gemm_path, s4_path, path, K):
    # -8 and 7 in every combination; K = 65536 is the largest K the in-kernel
    # conversion takes (its fp32 partial sums reach 225 K = 14.7e6 < 2^24)
    gemm_path(2)
    s4_path(path)
    A = np.full((512, K // 2), 0x88, dtype=np.uint8)   # rows 0..255: -8
    A[256:] = 0x77                                      # rows 256..511: 7
    B = np.full((512, K // 2), 0x88, dtype=np.uint8)
    B[256:] = 0x77
    C = _s4(dev, A, B, K)
    assert np.all(C[:256, :256] == 64 * K) and np.all(C[256:, 256:] == 49 * K)
    assert np.all(C[:256, 256:] == -56 * K) and np.all(C[256:, :256] == -56 * K)


@pytest.mark.parametrize("path", [0, 1])
@pytest.mark.parametrize("M,N,K", PATH_SHAPES + [(513, 777, 4160), (256, 512, 65568)])
def test_qgemm_s4_routes_on_pairs(dev, oracle, gemm_path, s4_path, path, M, N, K):
    # every shape on CTA pairs with either route; K = 65568 is past the
    # in-kernel conversion's limit, so route 0 falls back to the pre-pass
    gemm_path(2)
    s4_path(path)
    A = inputs.s4_packed_uniform(M, K, 1800 + M)
    B = inputs.s4_packed_uniform(N, K, 2800 + N)
    C = _s4(dev, A, B, K)
    if K > 8192:
        rows = inputs.sample_rows(M, 16, 4300 + M)
        ref = oracle.gemm_s4(A[rows], B, K)
        assert np.array_equal(C[rows], ref), first_mismatch(C[rows], ref)
    else:
        ref = oracle.gemm_s4(A, B, K)
        assert np.array_equal(C, ref), first_mismatch(C, ref)
