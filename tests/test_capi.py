"""CPU checks of the C ABI: the library loads, exports every declared symbol,
and rejects bad arguments synchronously (before touching any GPU)."""
import os

import pytest

import bit_quantized_tensor_gb300 as qg


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build_library()
    return qg.lib()


def test_exports_every_declared_symbol(L):
    names = qg.header_functions()
    assert len(names) >= 12
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    assert set(names) == set(qg.SIGNATURES)


def test_status_strings(L):
    for code, name in qg.STATUS_NAMES.items():
        assert L.qg_status_string(code).decode() == name
    assert L.qg_status_string(99).decode() == "QG_ERR_UNKNOWN"


def test_workspace_sizes(L):
    assert L.qg_workspace_size(qg.QG_OP_S8, 512, 512, 512) == 2 * 512 * 512 * 2
    assert L.qg_workspace_size(qg.QG_OP_S4, 100, 50, 64) == 6400 + 3328
    assert L.qg_workspace_size(qg.QG_OP_F16, 512, 512, 512) == 0
    assert L.qg_workspace_size(qg.QG_OP_S8, 0, 5, 5) == 0
    # host-memory INT8 GEMM: int8 A and B, their fp16 forms, int32 C with rows padded to 4
    # elements, each part at a 256-byte boundary
    r = lambda v: (v + 255) // 256 * 256  # noqa: E731
    M, N, K = 300, 5, 32
    assert L.qg_workspace_size(qg.QG_OP_S8_HOST, M, N, K) == \
        r(M * K) + r(N * K) + r(2 * M * K) + r(2 * N * K) + r(4 * M * 8)


FAKE = 0x10000  # a 16-byte aligned address that is never dereferenced
WS = 0x20000


def _s8(L, M=64, N=64, K=64, A=FAKE, lda=64, la=0, B=FAKE, ldb=64, lb=1, C=FAKE, ldc=64,
        ws=WS, wsb=1 << 30):
    return L.qgemm_s8(M, N, K, A, lda, la, B, ldb, lb, C, ldc, ws, wsb, None)


def test_qgemm_s8_argument_errors(L):
    assert _s8(L, M=0) == 1
    assert _s8(L, A=0) == 1
    assert _s8(L, K=40) == 1                 # K % 16
    assert _s8(L, lda=32) == 1               # lda < K
    assert _s8(L, la=1) == 2                 # layout
    assert _s8(L, lb=0) == 2
    assert _s8(L, A=FAKE + 8) == 3           # misaligned pointer
    assert _s8(L, lda=72) == 3               # lda not a multiple of 16 bytes
    assert _s8(L, wsb=10) == 4               # workspace too small
    assert _s8(L, ws=0) == 4
    assert _s8(L, ws=WS + 16) == 3           # workspace not 256-byte aligned


def test_gemm_f16_and_s4_argument_errors(L):
    assert L.gemm_f16(64, 64, 12, FAKE, 64, 0, FAKE, 64, 1, FAKE, 64, None) == 1
    assert L.gemm_f16(64, 64, 64, FAKE, 64, 0, FAKE, 64, 0, FAKE, 64, None) == 2
    assert L.gemm_f16(64, 64, 64, FAKE, 68, 0, FAKE, 64, 1, FAKE, 64, None) == 3
    assert L.qgemm_s4(64, 64, 48, FAKE, 32, 0, FAKE, 32, 1, FAKE, 64, WS, 1 << 30, None) == 1
    assert L.qgemm_s4(64, 64, 64, FAKE, 40, 0, FAKE, 32, 1, FAKE, 64, WS, 1 << 30, None) == 3


def test_no_gpu_reports_cuda_error(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _s8(L) == 5


def test_w4a16_and_w4a4_argument_errors(L):
    # w4a16_gemm(M, N, K, X, ldx, Wq, Wscale, group, Y, ldy, stream)
    assert L.w4a16_gemm(1, 64, 100, FAKE, 128, FAKE, FAKE, 128, FAKE, 64, None) == 1  # K % group
    assert L.w4a16_gemm(1, 64, 128, FAKE, 128, FAKE, FAKE, 64, FAKE, 64, None) == 2   # group
    assert L.w4a16_gemm(1, 64, 128, FAKE, 100, FAKE, FAKE, 128, FAKE, 64, None) == 1  # ldx < K
    assert L.w4a16_gemm(1, 64, 128, FAKE, 132, FAKE, FAKE, 128, FAKE, 64, None) == 3  # ldx % 8
    assert L.w4a16_gemm(1, 64, 128, FAKE + 2, 128, FAKE, FAKE, 128, FAKE, 64, None) == 3
    # w4a4_quantize(M, K, X, ldx, U, rank, Xq, Xs, XU, block, stream)
    assert L.w4a4_quantize(4, 96, FAKE, 96, None, 0, FAKE, FAKE, None, 64, None) == 1  # K % 64
    assert L.w4a4_quantize(4, 128, FAKE, 128, None, 0, FAKE, FAKE, None, 32, None) == 2
    assert L.w4a4_quantize(4, 128, FAKE, 128, FAKE, 16, FAKE, FAKE, FAKE, 64, None) == 2
    assert L.w4a4_quantize(4, 128, FAKE, 128, None, 32, FAKE, FAKE, FAKE, 64, None) == 1
    assert L.w4a4_quantize(4, 128, FAKE, 130, None, 0, FAKE, FAKE, None, 64, None) == 3
    # w4a4_gemm(M, N, K, Xq, Xs, Wq, Ws, block, XU, V, rank, bias, Y, ldy, ws, wsb, stream)
    big = 1 << 30
    assert L.w4a4_gemm(4, 8, 128, FAKE, FAKE, FAKE, FAKE, 32, None, None, 0, None, FAKE, 8,
                       WS, big, None) == 2
    assert L.w4a4_gemm(4, 8, 128, FAKE, FAKE, FAKE, FAKE, 64, None, None, 32, None, FAKE, 8,
                       WS, big, None) == 1
    assert L.w4a4_gemm(4, 8, 128, FAKE, FAKE, FAKE, FAKE, 64, None, None, 0, None, FAKE, 8,
                       WS, 16, None) == 4
    assert L.w4a4_gemm(4, 8, 128, FAKE, FAKE, FAKE, FAKE, 64, None, None, 0, None, FAKE, 4,
                       WS, big, None) == 1
    # w4a4_gemm_affine(M, N, K, Xq, Xs, Wq, Ws, block, XU, V, rank, alpha, bias, Y, ldy, ws, wsb, stream)
    assert L.w4a4_gemm_affine(4, 8, 128, FAKE, FAKE, FAKE, FAKE, 64, None, None, 0, None, None,
                              FAKE, 8, WS, big, None) == 1  # alpha is required
    assert L.w4a4_gemm_affine(4, 8, 128, FAKE, FAKE, FAKE, FAKE, 32, None, None, 0, FAKE, None,
                              FAKE, 8, WS, big, None) == 2
    assert L.w4a4_gemm_affine(4, 8, 128, FAKE, FAKE, FAKE, FAKE, 64, None, None, 0, FAKE, None,
                              FAKE, 8, WS, 16, None) == 4
    # w4a4_prepack_weights(N, K, Wq, Ws, block, alpha, packed, bytes, stream)
    assert L.w4a4_prepack_weights(8, 128, FAKE, FAKE, 32, None, WS, big, None) == 2
    assert L.w4a4_prepack_weights(8, 96, FAKE, FAKE, 64, None, WS, big, None) == 1
    assert L.w4a4_prepack_weights(8, 128, FAKE, FAKE, 64, None, WS, 16, None) == 4
    assert L.w4a4_prepack_weights(8, 128, FAKE, FAKE, 64, None, WS + 16, big, None) == 3
    # w4a4_gemm_prepacked(M, N, K, Xq, Xs, packed, bytes, block, XU, V, rank, bias, Y, ldy, ws, wsb, stream)
    assert L.w4a4_gemm_prepacked(4, 8, 128, FAKE, FAKE, WS, big, 64, None, None, 0, None, FAKE, 8,
                                 WS, 16, None) == 4
    assert L.w4a4_gemm_prepacked(4, 8, 128, FAKE, FAKE, WS, 16, 64, None, None, 0, None, FAKE, 8,
                                 WS, big, None) == 1
    assert L.qg_workspace_size(7, 1, 8, 128) < L.qg_workspace_size(4, 4, 8, 128)


def _s8h(L, M=64, N=64, K=64, A=FAKE, lda=64, B=FAKE, ldb=64, C=FAKE, ldc=64, ws=WS, wsb=1 << 30):
    return L.qgemm_s8_host(M, N, K, A, lda, B, ldb, C, ldc, ws, wsb, None)


def test_qgemm_s8_host_argument_errors(L):
    assert _s8h(L, M=0) == 1
    assert _s8h(L, N=-1) == 1
    assert _s8h(L, A=0) == 1
    assert _s8h(L, C=0) == 1
    assert _s8h(L, K=40) == 1                # K % 16
    assert _s8h(L, K=131072, lda=131072, ldb=131072) == 1
    assert _s8h(L, lda=32) == 1              # lda < K
    assert _s8h(L, ldc=63) == 1              # ldc < N
    assert _s8h(L, wsb=10) == 4              # workspace too small
    assert _s8h(L, ws=0) == 4
    assert _s8h(L, ws=WS + 16) == 3          # workspace not 256-byte aligned


def test_qgemm_s8_host_without_gpu_reports_cuda_error(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present (the fake host pointers would be read)")
    # host operands need no alignment: a valid call gets as far as the device
    assert _s8h(L, A=FAKE + 1, lda=65) == qg.QG_ERR_CUDA


def test_knob_ranges(L):
    # host-side setters: out-of-range values are refused, defaults restored
    assert L.qg_set_l2_policy(3) == 1 and L.qg_set_l2_policy(-1) == 1
    for m in (1, 2, 0):
        assert L.qg_set_l2_policy(m) == 0
    assert L.qg_set_gemm_path(3) == 1 and L.qg_set_gemm_path(0) == 0
    assert L.qg_set_s8_chunk(0) == 1 and L.qg_set_s8_chunk(17) == 1 and L.qg_set_s8_chunk(16) == 0


def test_product_package_never_touches_the_oracle():
    """The library's Python package and its C sources name no part of the
    CPU oracle: the product path has no CPU fallback to reach."""
    import re
    pkg = os.path.dirname(qg.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(root, f)).read()
                assert not re.search(r"\boracle\b|liboracle|qgemm_oracle", text), f


def test_binding_raises_without_its_library(tmp_path):
    """With the shared library absent the binding refuses to run (it does not
    fall back to anything)."""
    import subprocess
    import sys
    code = ("import bit_quantized_tensor_gb300 as qg\n"
            f"qg.LIB_PATH = {str(tmp_path / 'absent.so')!r}\n"
            "qg._lib = None\n"
            "try:\n"
            "    qg.lib()\n"
            "except Exception as e:\n"
            "    print('raised', type(e).__name__)\n"
            "else:\n"
            "    print('loaded')\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=os.path.dirname(os.path.dirname(__file__)),
                       capture_output=True, text=True, timeout=300)
    assert r.stdout.strip().startswith("raised"), r.stdout + r.stderr
