"""qgemm_s8_host on the GPU: operands and result in host memory, copies and
arithmetic overlapped inside the call.  Bit-exact against the oracle, with
several A slices and two B slices (ragged last slices), host row strides
larger than the rows, page-locked and pageable memory, a side stream, and
the full 8192-square shape on sampled rows."""
import numpy as np
import pytest

from bit_quantized_tensor_gb300 import inputs
from tests._util import first_mismatch

pytestmark = pytest.mark.gpu

SENTINEL = 0x5A5A5A5A


@pytest.fixture(scope="module")
def qg():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import bit_quantized_tensor_gb300 as qg
    qg.lib()
    return qg


@pytest.fixture(autouse=True)
def _status_clear(qg):
    yield
    assert qg.device_status() == qg.QG_OK


def _host(a, pinned, cols=None):
    """Host tensor holding `a`, optionally inside wider rows (cols >= a's)."""
    import torch
    cols = a.shape[1] if cols is None else cols
    buf = torch.zeros((a.shape[0], cols), dtype=torch.from_numpy(a[:0]).dtype)
    if pinned:
        buf = buf.pin_memory()
    buf[:, :a.shape[1]] = torch.from_numpy(a)
    return buf[:, :a.shape[1]]


def _out(M, N, ldc, pinned):
    import torch
    buf = torch.full((M, ldc), SENTINEL, dtype=torch.int32)
    if pinned:
        buf = buf.pin_memory()
    return buf, buf[:, :N]


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("M,N,K", [(2500, 4100, 64), (300, 260, 128), (1, 1, 16), (1100, 257, 48)])
def test_qgemm_s8_host_matches_oracle(qg, oracle, pinned, M, N, K):
    import torch
    A = inputs.s8_uniform(M, K, 4100 + M)
    B = inputs.s8_uniform(N, K, 4200 + N)
    Ah = _host(A, pinned, cols=K + 16)   # lda > K
    Bh = _host(B, pinned)
    buf, C = _out(M, N, N + 5, pinned)   # ldc > N
    qg.qgemm_s8_host(Ah, Bh, C=C)
    torch.cuda.synchronize()
    got, ref = C.numpy(), oracle.gemm_s8(A, B)
    assert np.array_equal(got, ref), first_mismatch(got, ref)
    assert np.all(buf.numpy()[:, N:] == SENTINEL), "columns past N were written"


def test_qgemm_s8_host_on_a_side_stream(qg, oracle):
    import torch
    M, N, K = 1500, 4400, 32
    A = inputs.s8_uniform(M, K, 4301)
    B = inputs.s8_uniform(N, K, 4302)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        C = qg.qgemm_s8_host(_host(A, True), _host(B, True), stream=s)
    s.synchronize()
    got, ref = C.numpy(), oracle.gemm_s8(A, B)
    assert np.array_equal(got, ref), first_mismatch(got, ref)
    # twice in a row into the same output: each call is ordered after the last
    A2 = inputs.s8_uniform(M, K, 4303)
    C2 = qg.qgemm_s8_host(_host(A2, True), _host(B, True), C=C, stream=s)
    s.synchronize()
    assert np.array_equal(C2.numpy(), oracle.gemm_s8(A2, B))


def test_qgemm_s8_host_full_size_sampled_rows(qg, oracle):
    import torch
    n, K = 8192, 512
    A = inputs.s8_uniform(n, K, 4401)
    B = inputs.s8_uniform(n, K, 4402)
    C = qg.qgemm_s8_host(_host(A, True), _host(B, True))
    torch.cuda.synchronize()
    rows = np.array([0, 1, 1023, 1024, 4095, 4096, 5000, 8191])
    got, ref = C.numpy()[rows], oracle.gemm_s8(A[rows], B)
    assert np.array_equal(got, ref), first_mismatch(got, ref)
    # every row and column: Freivalds' identity C.x == A.(B^T.x) in int64
    x = np.random.default_rng(7).integers(-3, 4, size=n).astype(np.int64)
    lhs = C.numpy().astype(np.int64) @ x
    rhs = A.astype(np.int64) @ (B.astype(np.int64).T @ x)
    assert np.array_equal(lhs, rhs)


def test_qgemm_s8_host_in_a_cuda_graph(qg, oracle):
    """Captured into a graph (the internal streams fork from the capturing
    stream and join back), then replayed with new host data in place."""
    import torch
    M, N, K = 1200, 4300, 32
    A = inputs.s8_uniform(M, K, 4501)
    B = inputs.s8_uniform(N, K, 4502)
    hA, hB = _host(A, True), _host(B, True)
    hC = torch.empty((M, N), dtype=torch.int32).pin_memory()
    ws = torch.empty(qg.workspace_size(qg.QG_OP_S8_HOST, M, N, K), dtype=torch.uint8, device="cuda")
    qg.qgemm_s8_host(hA, hB, C=hC, ws=ws)  # first call on the device creates the streams
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=s):
        qg.qgemm_s8_host(hA, hB, C=hC, ws=ws, stream=s)
    hC.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(hC.numpy(), oracle.gemm_s8(A, B))
    A2 = inputs.s8_uniform(M, K, 4503)
    hA.copy_(torch.from_numpy(A2))
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(hC.numpy(), oracle.gemm_s8(A2, B))
