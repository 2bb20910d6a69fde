"""qgemm_s8_noalloc: the INT8 GEMM for callers that cannot allocate.

Some callers of this library have no way to pass a workspace: plugin hosts
that give a kernel only its inputs and outputs, engines whose memory plan is
fixed after start-up, and code that must not call cudaMalloc at that point.
qgemm_s8_noalloc serves them from a 16 MiB static scratch array inside the
library.  These tests call it through the C ABI with raw device pointers and
compare its int32 result with qgemm_s8 given an ordinary workspace: integer
results must match exactly, on two calls in a row (the second call reuses
the scratch the first one left behind).  This file is collected last so that
a run stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest

import bit_quantized_tensor_gb300 as qg
from bit_quantized_tensor_gb300 import inputs


def _raw_call(A, B, C, stream):
    M, K = A.shape
    N = B.shape[0]
    return qg.lib().qgemm_s8_noalloc(M, N, K, A.data_ptr(), A.stride(0), qg.QG_ROW_MAJOR,
                                     B.data_ptr(), B.stride(0), qg.QG_COL_MAJOR,
                                     C.data_ptr(), C.stride(0), stream)


def test_scratch_need_at_the_documented_limit():
    # M = N = K = 2048 needs exactly the 16 MiB the array holds (two fp16
    # operand copies of 8 MiB each); K = 2064 needs 16 MiB + 128 KiB
    need = qg.lib().qg_workspace_size(qg.QG_OP_S8, 2048, 2048, 2048)
    assert need == 16 << 20
    assert qg.lib().qg_workspace_size(qg.QG_OP_S8, 2048, 2048, 2064) > 16 << 20


def test_rejects_problems_beyond_the_static_scratch():
    # 2*K*(M+N) = 2*4096*8192 = 64 MiB > 16 MiB: refused before any GPU work
    L = qg.lib()
    fake = 0x10000
    rc = L.qgemm_s8_noalloc(4096, 4096, 4096, fake, 4096, 0, fake, 4096, 1, fake, 4096, None)
    assert rc == 4  # QG_ERR_WORKSPACE


@pytest.mark.gpu
def test_matches_qgemm_s8_on_two_calls_in_a_row():
    import torch
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream().cuda_stream
    shapes = [(1000, 1100, 2048), (333, 2048, 1040)]   # 2*K*(M+N) <= 16 MiB each
    for i, (M, N, K) in enumerate(shapes):
        A = torch.from_numpy(inputs.s8_uniform(M, K, 7000 + i)).to(dev)
        B = torch.from_numpy(inputs.s8_uniform(N, K, 8000 + i)).to(dev)
        C = torch.full((M, N), -1, dtype=torch.int32, device=dev)
        assert qg.lib().qg_workspace_size(qg.QG_OP_S8, M, N, K) <= 16 << 20
        assert _raw_call(A, B, C, stream) == qg.QG_OK
        ref = qg.qgemm_s8(A, B)           # the existing entry point, with a workspace
        torch.cuda.synchronize()
        got, want = C.cpu().numpy(), ref.cpu().numpy()
        assert np.array_equal(got, want), f"call {i}: noalloc result differs from qgemm_s8"
    assert qg.device_status() == qg.QG_OK


@pytest.mark.gpu
def test_the_largest_accepted_and_the_smallest_refused_problem():
    import torch
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream().cuda_stream
    # exactly the array's size: accepted, bit-exact against qgemm_s8
    A = torch.from_numpy(inputs.s8_uniform(2048, 2048, 7100)).to(dev)
    B = torch.from_numpy(inputs.s8_uniform(2048, 2048, 8100)).to(dev)
    C = torch.full((2048, 2048), -1, dtype=torch.int32, device=dev)
    assert _raw_call(A, B, C, stream) == qg.QG_OK
    ref = qg.qgemm_s8(A, B)
    torch.cuda.synchronize()
    assert torch.equal(C, ref)
    # 16 more k values: refused before anything is enqueued, C untouched
    A2 = torch.from_numpy(inputs.s8_uniform(2048, 2064, 7101)).to(dev)
    B2 = torch.from_numpy(inputs.s8_uniform(2048, 2064, 8101)).to(dev)
    C2 = torch.full((2048, 2048), 12345, dtype=torch.int32, device=dev)
    assert _raw_call(A2, B2, C2, stream) == qg.QG_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((C2 == 12345).all())
    assert qg.device_status() == qg.QG_OK
