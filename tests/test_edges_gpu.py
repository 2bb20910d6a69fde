"""Edge cases of the persistent tile schedulers and of output bounds, on the GPU.

- Tile counts just below, at and above the number of CTAs (one-CTA kernels)
  or CTA pairs (paired kernels) that the persistent schedulers run: the last
  round of tiles is partial, full, or one tile over, or just under and just
  over half full.
- Guard regions: every output is a view inside a larger buffer filled with a
  sentinel pattern, with a row stride larger than N; after the call the rows
  above and below and the columns past N must still hold the sentinel, and
  the view must match the oracle.
- Strided inputs: every input that takes a leading dimension is read as the
  first K columns of a wider buffer (whose extra columns hold values that
  would change the result if they were read).
"""
import numpy as np
import pytest

from bit_quantized_tensor_gb300 import inputs
from tests._util import assert_fp16_close, first_mismatch

pytestmark = pytest.mark.gpu

GROUP = 128
BLOCK = 64
SENTINEL_I32 = 0x5A5A5A5A
SENTINEL_F16 = 0x5A5A  # bit pattern of 203.25 in fp16


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


@pytest.fixture
def gemm_path():
    import bit_quantized_tensor_gb300 as qg

    def set_path(p):
        assert qg.lib().qg_set_gemm_path(p) == 0
    yield set_path
    qg.lib().qg_set_gemm_path(0)


def _t(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def _sms():
    import torch
    return torch.cuda.get_device_properties(0).multi_processor_count


def _factor(T):
    """Tile grid a x b with a * b == T and a as close to sqrt(T) as possible."""
    a = int(np.sqrt(T))
    while T % a:
        a -= 1
    return a, T // a


# ------------------------------------------------------- tile-count sweeps

def _sweep_counts(units):
    # around one round; one over two rounds; a last round a little under and
    # a little over half full
    return sorted({max(1, units - 1), units, units + 1, 2 * units + 1,
                   units + units // 2 - 1, units + units // 2 + 1})


@pytest.mark.parametrize("which", range(6))
@pytest.mark.parametrize("path,bm,bn,per", [(1, 128, 256, 1), (2, 256, 256, 2)])
def test_qgemm_s8_tile_counts_around_the_grid(dev, oracle, gemm_path, which, path, bm, bn, per):
    """qgemm_s8 on the one-CTA kernel (128 x 256 tiles, one CTA per SM) and
    the paired kernel (256 x 256 tiles per pair, two SMs per pair), with
    ragged edges, at tile counts around the resident grid."""
    import bit_quantized_tensor_gb300 as qg
    gemm_path(path)
    counts = _sweep_counts(_sms() // per)
    if which >= len(counts):
        pytest.skip("fewer distinct tile counts on this device")
    T = counts[which]
    a, b = _factor(T)
    M, N, K = a * bm - 3, b * bn - 5, 64 if path == 1 else 320
    if path == 2 and (M < 256 or N < 256):  # pairs need two row blocks' worth
        M, N = max(M, 256), max(N, 256)
    A = inputs.s8_uniform(M, K, 1500 + T)
    B = inputs.s8_uniform(N, K, 2500 + T)
    C = qg.qgemm_s8(_t(A, dev), _t(B, dev)).cpu().numpy()
    ref = oracle.gemm_s8(A, B)
    assert np.array_equal(C, ref), f"T={T} ({M}x{N}): " + first_mismatch(C, ref)


# ------------------------------------------------------------ guard regions

def _guarded(M, N, dtype, dev):
    """(buffer, view): the view is rows 1..M, columns 0..N-1 of a buffer with
    two guard rows and a row stride past N (a multiple of 8 elements, so every
    row starts 16-byte aligned)."""
    import torch
    ld = (N + 13 + 7) // 8 * 8
    if dtype == torch.int32:
        buf = torch.full((M + 2, ld), SENTINEL_I32, dtype=torch.int32, device=dev)
    else:
        buf = torch.full((M + 2, ld), SENTINEL_F16, dtype=torch.int16, device=dev).view(torch.float16)
    return buf, buf[1:M + 1, :N]


def _check_guards(buf, M, N):
    import torch
    raw = buf.view(torch.int32) if buf.dtype == torch.int32 else buf.view(torch.int16)
    want = SENTINEL_I32 if buf.dtype == torch.int32 else SENTINEL_F16
    raw = raw.cpu().numpy()
    assert np.all(raw[0] == want), "row above the output was written"
    assert np.all(raw[M + 1] == want), "row below the output was written"
    assert np.all(raw[1:M + 1, N:] == want), "columns past N were written"


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("M,N,K", [(1, 3, 16), (257, 263, 144), (300, 520, 1040)])
def test_qgemm_s8_writes_only_its_output(dev, oracle, gemm_path, path, M, N, K):
    import torch
    import bit_quantized_tensor_gb300 as qg
    gemm_path(path)
    A = inputs.s8_uniform(M, K, 1600 + M)
    B = inputs.s8_uniform(N, K, 2600 + N)
    buf, C = _guarded(M, N, torch.int32, dev)
    qg.qgemm_s8(_t(A, dev), _t(B, dev), C=C)
    torch.cuda.synchronize()
    _check_guards(buf, M, N)
    got, ref = C.cpu().numpy(), oracle.gemm_s8(A, B)
    assert np.array_equal(got, ref), first_mismatch(got, ref)


@pytest.mark.parametrize("path", [1, 2])
def test_qgemm_s4_writes_only_its_output(dev, oracle, gemm_path, path):
    import torch
    import bit_quantized_tensor_gb300 as qg
    gemm_path(path)
    M, N, K = 261, 300, 96
    A = inputs.s4_packed_uniform(M, K, 1700)
    B = inputs.s4_packed_uniform(N, K, 2700)
    buf, C = _guarded(M, N, torch.int32, dev)
    qg.qgemm_s4(_t(A, dev), _t(B, dev), K, C=C)
    torch.cuda.synchronize()
    _check_guards(buf, M, N)
    got, ref = C.cpu().numpy(), oracle.gemm_s4(A, B, K)
    assert np.array_equal(got, ref), first_mismatch(got, ref)


@pytest.mark.parametrize("path", [1, 2])
def test_gemm_f16_writes_only_its_output(dev, oracle, gemm_path, path):
    import torch
    import bit_quantized_tensor_gb300 as qg
    gemm_path(path)
    M, N, K = 259, 270, 88
    A = inputs.f16_normal(M, K, 1800)
    B = inputs.f16_normal(N, K, 2800)
    buf, C = _guarded(M, N, torch.float16, dev)
    qg.gemm_f16(_t(A, dev), _t(B, dev), C=C)
    torch.cuda.synchronize()
    _check_guards(buf, M, N)
    assert_fp16_close(C.cpu().numpy(), oracle.gemm_f16(A, B), "gemm_f16 guarded")


def _guarded_16(M, N, dtype, dev):
    """Like _guarded, but the row stride is 16 bytes past a multiple of 32:
    the rows alternate between 32-byte aligned starts (32-byte stores) and
    starts that are 16-byte aligned only (16-byte stores)."""
    import torch
    esz = 4 if dtype == torch.int32 else 2
    ld = (N + 13 + 15) // 16 * 16 + 16 // esz
    assert (ld * esz) % 32 == 16
    if dtype == torch.int32:
        buf = torch.full((M + 2, ld), SENTINEL_I32, dtype=torch.int32, device=dev)
    else:
        buf = torch.full((M + 2, ld), SENTINEL_F16, dtype=torch.int16, device=dev).view(torch.float16)
    return buf, buf[1:M + 1, :N]


@pytest.mark.parametrize("path", [1, 2])
def test_gemm_outputs_with_16_byte_row_alignment(dev, oracle, gemm_path, path):
    import torch
    import bit_quantized_tensor_gb300 as qg
    gemm_path(path)
    M, N, K = 300, 299, 160
    A = inputs.s8_uniform(M, K, 1900)
    B = inputs.s8_uniform(N, K, 2900)
    buf, C = _guarded_16(M, N, torch.int32, dev)
    qg.qgemm_s8(_t(A, dev), _t(B, dev), C=C)
    torch.cuda.synchronize()
    _check_guards(buf, M, N)
    got, ref = C.cpu().numpy(), oracle.gemm_s8(A, B)
    assert np.array_equal(got, ref), "s8: " + first_mismatch(got, ref)

    A4 = inputs.s4_packed_uniform(M, K, 1901)
    B4 = inputs.s4_packed_uniform(N, K, 2901)
    buf, C = _guarded_16(M, N, torch.int32, dev)
    qg.qgemm_s4(_t(A4, dev), _t(B4, dev), K, C=C)
    torch.cuda.synchronize()
    _check_guards(buf, M, N)
    got, ref = C.cpu().numpy(), oracle.gemm_s4(A4, B4, K)
    assert np.array_equal(got, ref), "s4: " + first_mismatch(got, ref)

    Ah = inputs.f16_normal(M, K, 1902)
    Bh = inputs.f16_normal(N, K, 2902)
    buf, C = _guarded_16(M, N, torch.float16, dev)
    qg.gemm_f16(_t(Ah, dev), _t(Bh, dev), C=C)
    torch.cuda.synchronize()
    _check_guards(buf, M, N)
    assert_fp16_close(C.cpu().numpy(), oracle.gemm_f16(Ah, Bh), "gemm_f16 16-byte rows")


# M = 1 and 5: GEMV with staged X; 12: GEMV with X from L2; 130: tensor-core
# path with a ragged second launch of 2 rows
@pytest.mark.parametrize("M,N,K", [(1, 4100, 512), (5, 300, 1024), (12, 2000, 768), (130, 260, 512)])
def test_w4a16_writes_only_its_output(dev, oracle, M, N, K):
    import torch
    import bit_quantized_tensor_gb300 as qg
    X = inputs.f16_normal(M, K, 1900 + M)
    Wq = inputs.s4_packed_uniform(N, K, 2900 + M)
    S = inputs.f16_uniform(N, K // GROUP, 0.005, 0.02, 3900 + M)
    buf, Y = _guarded(M, N, torch.float16, dev)
    qg.w4a16_gemm(_t(X, dev), _t(Wq, dev), _t(S, dev), GROUP, Y=Y)
    torch.cuda.synchronize()
    _check_guards(buf, M, N)
    assert_fp16_close(Y.cpu().numpy(), oracle.w4a16(X, Wq, S, GROUP), f"w4a16 guarded {M}x{N}x{K}")


@pytest.mark.parametrize("path", [1, 2])
def test_w4a4_gemm_writes_only_its_output(dev, oracle, gemm_path, path):
    import torch
    import bit_quantized_tensor_gb300 as qg
    gemm_path(path)
    M, N, K, R = 260, 200, 256, 32
    X = inputs.f32_normal(M, K, 1950)
    W = inputs.f32_normal(N, K, 2950)
    U = inputs.f16_normal(K, R, 3950, sigma=0.02)
    V = inputs.f16_normal(R, N, 3960, sigma=0.02)
    b = inputs.f16_normal(1, N, 3970, sigma=0.1)[0]
    qx, sx = oracle.w4a4_quantize(X, BLOCK)
    qw, sw = oracle.w4a4_quantize(W, BLOCK)
    xu16 = oracle.lowrank_xu(X, U).astype(np.float16)
    buf, Y = _guarded(M, N, torch.float16, dev)
    qg.w4a4_gemm(_t(qx, dev), _t(sx.view(np.float16), dev), _t(qw, dev), _t(sw.view(np.float16), dev),
                 K, XU=_t(xu16, dev), Vt=_t(V.T, dev), bias=_t(b, dev), Y=Y)
    torch.cuda.synchronize()
    _check_guards(buf, M, N)
    ref = oracle.w4a4_gemm(qx, sx, qw, sw, BLOCK, K, XU=xu16.astype(np.float64), V=V, bias=b)
    assert_fp16_close(Y.cpu().numpy(), ref, "w4a4 guarded")


# ---------------------------------------------------------- strided inputs

def _wide(a, extra, fill):
    """a as the left columns of a wider array whose other columns hold `fill`."""
    w = np.full((a.shape[0], a.shape[1] + extra), fill, dtype=a.dtype)
    w[:, :a.shape[1]] = a
    return w


@pytest.mark.parametrize("path", [1, 2])
def test_gemms_read_inputs_through_leading_dimensions(dev, oracle, gemm_path, path):
    import bit_quantized_tensor_gb300 as qg
    gemm_path(path)
    M, N, K = 300, 520, 1104
    A = inputs.s8_uniform(M, K, 4100)
    B = inputs.s8_uniform(N, K, 4101)
    tA, tB = _t(_wide(A, 48, 127), dev)[:, :K], _t(_wide(B, 32, -128), dev)[:, :K]
    assert tA.stride(0) == K + 48 and tB.stride(0) == K + 32
    C = qg.qgemm_s8(tA, tB).cpu().numpy()
    ref = oracle.gemm_s8(A, B)
    assert np.array_equal(C, ref), first_mismatch(C, ref)

    K4 = 1088  # a multiple of 32; rows of 544 bytes, strides of 560 and 592
    A4 = inputs.s4_packed_uniform(M, K4, 4102)
    B4 = inputs.s4_packed_uniform(N, K4, 4103)
    tA4 = _t(_wide(A4, 16, 0x77), dev)[:, :K4 // 2]
    tB4 = _t(_wide(B4, 48, 0x88), dev)[:, :K4 // 2]
    C4 = qg.qgemm_s4(tA4, tB4, K4).cpu().numpy()
    ref4 = oracle.gemm_s4(A4, B4, K4)
    assert np.array_equal(C4, ref4), first_mismatch(C4, ref4)

    Af = inputs.f16_normal(M, K, 4104)
    Bf = inputs.f16_normal(N, K, 4105)
    Cf = qg.gemm_f16(_t(_wide(Af, 8, np.float16(1000)), dev)[:, :K],
                     _t(_wide(Bf, 24, np.float16(-1000)), dev)[:, :K]).cpu().numpy()
    assert_fp16_close(Cf, oracle.gemm_f16(Af, Bf), "gemm_f16 strided inputs")


@pytest.mark.parametrize("M", [1, 12, 40])
def test_w4a16_reads_x_through_its_leading_dimension(dev, oracle, M):
    """Decode GEMV (M=1), batched GEMV (M=12) and the tensor-core path (M=40)."""
    import bit_quantized_tensor_gb300 as qg
    N, K = 700, 1024
    X = inputs.f16_normal(M, K, 4110 + M)
    Wq = inputs.s4_packed_uniform(N, K, 4120 + M)
    S = inputs.f16_uniform(N, K // GROUP, 0.005, 0.02, 4130 + M)
    tX = _t(_wide(X, 64, np.float16(500)), dev)[:, :K]
    assert tX.stride(0) == K + 64
    Y = qg.w4a16_gemm(tX, _t(Wq, dev), _t(S, dev), GROUP).cpu().numpy()
    assert_fp16_close(Y, oracle.w4a16(X, Wq, S, GROUP), f"w4a16 strided X M={M}")


def test_w4a4_quantize_reads_x_through_its_leading_dimension(dev, oracle):
    import bit_quantized_tensor_gb300 as qg
    M, K = 70, 576
    X = inputs.f32_normal(M, K, 4140)
    tX = _t(_wide(X, 20, np.float32(1e6)), dev)[:, :K]
    assert tX.stride(0) == K + 20
    q, sc, _ = qg.w4a4_quantize(tX, None, BLOCK)
    q_ref, s_ref = oracle.w4a4_quantize(X, BLOCK)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(sc.cpu().numpy().view(np.uint16), s_ref)
