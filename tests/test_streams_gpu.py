"""Concurrency and graph capture on the GPU.

- Several host threads, each with its own CUDA stream and its own outputs and
  workspaces, call the library at the same time: every result must match the
  oracle (the calls are documented as thread-safe; the per-device set-up the
  library does on first use is guarded by locks).
- Every device-memory entry point captured into a CUDA graph and replayed
  twice gives the oracle's result each time.
"""
import threading

import numpy as np
import pytest

from bit_quantized_tensor_gb300 import inputs
from tests._util import assert_fp16_close, first_mismatch

pytestmark = pytest.mark.gpu

GROUP = 128
BLOCK = 64


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


def _cases(dev, seed):
    """One small problem per operation: (name, run(stream) -> numpy result, check)."""
    import bit_quantized_tensor_gb300 as qg
    out = []
    A = inputs.s8_uniform(300, 1040, seed)
    B = inputs.s8_uniform(260, 1040, seed + 1)
    tA, tB = _t(A, dev), _t(B, dev)
    ref8 = None

    def s8(stream):
        return qg.qgemm_s8(tA, tB, stream=stream)

    def chk8(got):
        nonlocal ref8
        import oracle
        ref8 = oracle.gemm_s8(A, B) if ref8 is None else ref8
        assert np.array_equal(got, ref8), first_mismatch(got, ref8)
    out.append(("qgemm_s8", s8, chk8))

    X = inputs.f16_normal(3, 768, seed + 2)
    Wq = inputs.s4_packed_uniform(500, 768, seed + 3)
    S = inputs.f16_uniform(500, 768 // GROUP, 0.005, 0.02, seed + 4)
    tX, tW, tS = _t(X, dev), _t(Wq, dev), _t(S, dev)

    def w16(stream):
        return qg.w4a16_gemm(tX, tW, tS, GROUP, stream=stream)

    def chk16(got):
        import oracle
        assert_fp16_close(got, oracle.w4a16(X, Wq, S, GROUP), "w4a16 concurrent")
    out.append(("w4a16_gemm", w16, chk16))

    Xf = inputs.f32_normal(140, 512, seed + 5)
    Wf = inputs.f32_normal(200, 512, seed + 6)
    tXf = _t(Xf, dev)
    qw, sw, _ = qg.w4a4_quantize(_t(Wf, dev), None, BLOCK)

    def w4(stream):
        q, s, _ = qg.w4a4_quantize(tXf, None, BLOCK, stream=stream)
        return qg.w4a4_gemm(q, s, qw, sw, 512, stream=stream)

    def chk4(got):
        import oracle
        qx, sx = oracle.w4a4_quantize(Xf, BLOCK)
        qwr, swr = oracle.w4a4_quantize(Wf, BLOCK)
        assert_fp16_close(got, oracle.w4a4_gemm(qx, sx, qwr, swr, BLOCK, 512), "w4a4 concurrent")
    out.append(("w4a4", w4, chk4))
    return out


def test_threads_on_their_own_streams(dev):
    import torch
    errors, results = [], {}
    cases = _cases(dev, 5000)

    def worker(i):
        try:
            torch.cuda.set_device(dev)
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                for _ in range(3):
                    for name, run, _ in cases:
                        y = run(stream)
                        stream.synchronize()
                        results[(i, name)] = y.cpu().numpy()
        except Exception as e:  # reported on the main thread
            errors.append(f"thread {i}: {e!r}")

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=120)
    assert not errors, errors
    for i in range(4):
        for name, _, check in cases:
            check(results[(i, name)])


def test_graph_capture_and_replay(dev):
    import torch
    import bit_quantized_tensor_gb300 as qg
    torch.cuda.synchronize()
    cases = _cases(dev, 5100)
    stream = torch.cuda.Stream()
    outs = {}
    with torch.cuda.stream(stream):
        for name, run, _ in cases:  # first calls outside the capture (one-time set-up)
            run(stream)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for name, run, _ in cases:
                outs[name] = run(stream)
    for _ in range(2):
        for y in outs.values():
            y.zero_()
        g.replay()
        torch.cuda.synchronize()
        for name, _, check in cases:
            check(outs[name].cpu().numpy())
    assert qg.device_status() == qg.QG_OK
