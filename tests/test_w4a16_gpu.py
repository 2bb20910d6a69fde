"""GPU parity of w4a16_gemm against the CPU oracle (dequantize, then FP64 GEMM)."""
import numpy as np
import pytest

from bit_quantized_tensor_gb300 import inputs
from tests._util import assert_fp16_close

pytestmark = pytest.mark.gpu

GROUP = 128


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


def _operands(M, N, K, idx=3):
    X = inputs.f16_normal(M, K, 1000 + idx)
    Wq = inputs.s4_packed_uniform(N, K, 2000 + idx)
    S = inputs.f16_uniform(N, K // GROUP, 0.005, 0.02, 3000 + idx)
    return X, Wq, S


def _run(dev, X, Wq, S):
    import bit_quantized_tensor_gb300 as qg
    return qg.w4a16_gemm(_t(X, dev), _t(Wq, dev), _t(S, dev), GROUP).cpu().numpy()


@pytest.mark.parametrize("M", [1, 16, 128])
def test_w4a16_4096(dev, oracle, M):
    X, Wq, S = _operands(M, 4096, 4096)
    assert_fp16_close(_run(dev, X, Wq, S), oracle.w4a16(X, Wq, S, GROUP), f"w4a16 M={M}")


@pytest.mark.parametrize("M,N,K", [(1, 8, 128), (1, 1, 128), (3, 100, 256), (17, 260, 384),
                                   (40, 72, 1024), (77, 333, 640), (130, 48, 256),
                                   (9, 4096, 11008 // 128 * 128), (2, 64, 8192),
                                   (1, 40, 16384), (12, 40, 20480), (1, 24, 20480),
                                   (5, 33, 24576), (8, 5000, 2048), (16, 3001, 1152),
                                   (7, 300, 4096), (13, 4864, 512)])
def test_w4a16_shapes(dev, oracle, M, N, K):
    X, Wq, S = _operands(M, N, K, idx=M + N)
    assert_fp16_close(_run(dev, X, Wq, S), oracle.w4a16(X, Wq, S, GROUP), f"w4a16 {M}x{N}x{K}")


def test_w4a16_unit_scale_integer_inputs_exact(dev, oracle):
    # integer X in [-2, 2], scale 1: every partial sum is an integer of
    # magnitude <= 2 * 8 * 128 = 2048, exact in fp32 and in the fp16 output.
    M, N, K = 16, 96, 128
    X = inputs.s8_in_range(M, K, -2, 2, 10).astype(np.float16)
    Wq = inputs.s4_packed_uniform(N, K, 11)
    S = np.ones((N, 1), dtype=np.float16)
    Y = _run(dev, X, Wq, S)
    assert np.array_equal(Y.astype(np.float64), oracle.w4a16(X, Wq, S, GROUP))


def test_w4a16_group_scales_are_per_row_and_group(dev, oracle):
    # scales that differ by orders of magnitude across rows and groups expose
    # any transposed or shifted scale index
    M, N, K = 4, 40, 512
    X, Wq, _ = _operands(M, N, K, idx=12)
    S = (2.0 ** inputs.s8_in_range(N, K // GROUP, -8, 4, 13)).astype(np.float16)
    assert_fp16_close(_run(dev, X, Wq, S), oracle.w4a16(X, Wq, S, GROUP), "w4a16 pow2 scales")


@pytest.mark.parametrize("M,N,K", [(17, 260, 384), (130, 48, 256), (40, 72, 1024), (128, 4096, 4096),
                                   (200, 520, 3968), (33, 128, 4224), (64, 256, 8192)])
def test_w4a16_tc_forms_identical(dev, oracle, M, N, K):
    """The tensor-core kernel with every packed row of a K quarter resident
    (K <= 4096, the default there) and the ring form give the same bits;
    K = 4224 and 8192 exceed the resident form and run the ring form both
    times."""
    import bit_quantized_tensor_gb300 as qg
    X, Wq, S = _operands(M, N, K, idx=M + K)
    try:
        got = {}
        for form in (0, 1):
            assert qg.lib().qg_set_w4a16_tc_form(form) == qg.QG_OK
            got[form] = _run(dev, X, Wq, S)
    finally:
        qg.lib().qg_set_w4a16_tc_form(0)
    assert np.array_equal(got[0].view(np.uint16), got[1].view(np.uint16))
    assert_fp16_close(got[0], oracle.w4a16(X, Wq, S, GROUP), f"w4a16 tc {M}x{N}x{K}")


@pytest.mark.parametrize("M", [1, 12, 32, 128])
@pytest.mark.parametrize("pdl", [1, 0])
def test_w4a16_chain_reads_previous_output(dev, oracle, pdl, M):
    """Layer chain Y_i = f_i(Y_{i-1}) on one stream: with programmatic
    dependent launch each kernel streams its weights early but must read X
    only after the previous kernel finished.  The scales keep activations at
    the same magnitude from layer to layer (|q| averages 4.6, so s ~ 1 /
    sqrt(K * E[q^2]) ~ 0.0067), as normalization does in a network; with
    activations growing 4x per layer the last layer's near-zero outputs would
    test fp32 accumulation over 1e4-sized terms rather than the ordering."""
    import torch
    import bit_quantized_tensor_gb300 as qg
    N = K = 1024
    layers = [(inputs.s4_packed_uniform(N, K, 2100 + i),
               inputs.f16_uniform(N, K // GROUP, 0.005, 0.008, 3100 + i)) for i in range(4)]
    X0 = inputs.f16_normal(M, K, 1100)
    qg.lib().qg_set_pdl(pdl)
    try:
        x = _t(X0, dev)
        dW = [(_t(w, dev), _t(s, dev)) for w, s in layers]
        for w, s in dW:
            x = qg.w4a16_gemm(x, w, s, GROUP)
        torch.cuda.synchronize()
        got = x.cpu().numpy()
    finally:
        qg.lib().qg_set_pdl(1)
    ref = X0
    for w, s in layers:
        ref = oracle.w4a16(ref, w, s, GROUP).astype(np.float16)
    assert_fp16_close(got, ref.astype(np.float64), f"w4a16 chain M={M} pdl={pdl}")


@pytest.mark.parametrize("M,N,K", [(9, 1000, 4608), (16, 300, 2048), (11, 4096, 4096), (16, 152, 128),
                                   (14, 5000, 1024), (10, 33, 3968)])
def test_w4a16_batched_gemv_shapes(dev, oracle, M, N, K):
    """9 <= M <= 16: ragged N, unrolled and generic group loops, one and two
    m16 tiles per CTA."""
    X, Wq, S = _operands(M, N, K, idx=M + 3 * N)
    assert_fp16_close(_run(dev, X, Wq, S), oracle.w4a16(X, Wq, S, GROUP), f"w4a16 {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(1, 4096, 8192), (1, 4096, 11008), (4, 4096, 8192), (8, 4096, 4096),
                                   (1, 3000, 16384), (2, 4100, 8320)])
def test_w4a16_gemv_large_slabs(dev, oracle, M, N, K):
    """Decode shapes whose weight slab per SM does not fit at half an SM
    (fewer rows per CTA, more CTAs than SMs)."""
    X, Wq, S = _operands(M, N, K, idx=M + 7 * N)
    assert_fp16_close(_run(dev, X, Wq, S), oracle.w4a16(X, Wq, S, GROUP), f"w4a16 {M}x{N}x{K}")


@pytest.mark.parametrize("pdl", [1, 0])
def test_w4a16_chain_of_large_layers(dev, oracle, pdl):
    """A chain of N = K = 8192 decode layers (M = 1, more CTAs than SMs): each
    call reads X only after the previous call has finished."""
    import torch
    import bit_quantized_tensor_gb300 as qg
    N = K = 8192
    layers = [(inputs.s4_packed_uniform(N, K, 2400 + i),
               inputs.f16_uniform(N, K // GROUP, 0.0035, 0.0055, 3400 + i)) for i in range(3)]
    X0 = inputs.f16_normal(1, K, 1400)
    qg.lib().qg_set_pdl(pdl)
    try:
        x = _t(X0, dev)
        dW = [(_t(w, dev), _t(s, dev)) for w, s in layers]
        for w, s in dW:
            x = qg.w4a16_gemm(x, w, s, GROUP)
        torch.cuda.synchronize()
        got = x.cpu().numpy()
    finally:
        qg.lib().qg_set_pdl(1)
    ref = X0
    for w, s in layers:
        ref = oracle.w4a16(ref, w, s, GROUP).astype(np.float16)
    assert_fp16_close(got, ref.astype(np.float64), f"w4a16 large chain pdl={pdl}")
