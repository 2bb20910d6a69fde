"""Python binding of libqgemm.so, the GB300 quantized tensor-core GEMM library.

Argument marshalling only: every step of every operation runs in the CUDA
kernels behind the C ABI declared in ``include/qgemm.h``.  PyTorch supplies
device memory and the current CUDA stream.  There is no fallback: if the
library is not built, or the tensors are not CUDA tensors, the calls raise.

Functions (same names as the C ABI):
  qgemm_s8(A, B)            exact int8 GEMM,  A: M x K int8, B: N x K int8 -> int32 M x N
  qgemm_s4(A, B, K)         exact int4 GEMM on packed operands (M x K/2, N x K/2 uint8)
  gemm_f16(A, B)            fp16 GEMM with fp32 accumulation -> fp16 M x N
  w4a16_gemm(X, Wq, Wscale) weight-only INT4 linear, per-group (128) fp16 scales
  w4a4_quantize(X, U)       per-row, per-64-block absmax INT4 quantizer (+ X.U)
  w4a4_gemm(...)            Y = (Q(X).Q(W)^T) (.) scale + (X.U).V + b
                            (alpha=...: the column-wise affine form,
                            Y = alpha (.) (...) + b, through w4a4_gemm_affine)
B / W operands are K-major (N x K row-major), the layout every call takes.
"""
from __future__ import annotations

import ctypes
import os
import re

from . import inputs  # noqa: F401  (seeded input generators)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqgemm.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "qgemm.h")

(QG_OK, QG_ERR_INVALID_ARG, QG_ERR_UNSUPPORTED, QG_ERR_MISALIGNED, QG_ERR_WORKSPACE, QG_ERR_CUDA,
 QG_ERR_TIMEOUT) = range(7)
STATUS_NAMES = {0: "QG_OK", 1: "QG_ERR_INVALID_ARG", 2: "QG_ERR_UNSUPPORTED",
                3: "QG_ERR_MISALIGNED", 4: "QG_ERR_WORKSPACE", 5: "QG_ERR_CUDA",
                6: "QG_ERR_TIMEOUT"}
QG_ROW_MAJOR, QG_COL_MAJOR = 0, 1
(QG_OP_S8, QG_OP_S4, QG_OP_F16, QG_OP_W4A16, QG_OP_W4A4, QG_OP_S8_HOST, QG_OP_W4A4_PREPACKED,
 QG_OP_W4A4_WEIGHTS) = range(8)


class QgError(RuntimeError):
    def __init__(self, name: str, code: int):
        super().__init__(f"{name} failed: {STATUS_NAMES.get(code, code)}")
        self.code = code


class KernelBudgetC(ctypes.Structure):
    """qg_kernel_budget of the C ABI."""
    _fields_ = [("kernel", ctypes.c_char_p), ("threads", ctypes.c_int), ("smem_bytes", ctypes.c_int),
                ("tmem_cols", ctypes.c_int), ("cluster", ctypes.c_int), ("min_ctas_per_sm", ctypes.c_int)]


_i64 = ctypes.c_int64
_p = ctypes.c_void_p
_sz = ctypes.c_size_t
_int = ctypes.c_int

# C signatures (restype, argtypes) of every exported function.
SIGNATURES = {
    "qg_status_string": (ctypes.c_char_p, [_int]),
    "qg_version": (_int, []),
    "qg_workspace_size": (_sz, [_int, _i64, _i64, _i64]),
    "qg_device_status": (_int, [_p]),
    "qg_device_status_detail": (_int, [ctypes.POINTER(ctypes.c_int), _p]),
    "qg_last_cuda_error": (_int, []),
    "qg_set_timeout_ns": (_int, [ctypes.c_uint64]),
    "qg_selftest_wait_timeout": (_int, [ctypes.c_uint64, _p]),
    "qg_selftest_deadlock": (_int, [_int, ctypes.c_uint64, _p]),
    "qg_kernel_budget_count": (_int, []),
    "qg_kernel_budget_get": (_int, [_int, ctypes.POINTER(KernelBudgetC)]),
    "qg_kernel_budget_measure": (_int, [_int, ctypes.POINTER(_int), ctypes.POINTER(_int), ctypes.POINTER(_int)]),
    "qg_set_s8_chunk": (_int, [_int]),
    "qg_set_gemm_path": (_int, [_int]),
    "qg_set_s4_path": (_int, [_int]),
    "qg_set_w4a4_pair_form": (_int, [_int]),
    "qg_set_l2_policy": (_int, [_int]),
    "qg_set_pdl": (_int, [_int]),
    "qg_set_w4a16_tc_form": (_int, [_int]),
    "qg_set_profile_events": (_int, [_p, _p]),
    "qgemm_s8": (_int, [_i64, _i64, _i64, _p, _i64, _int, _p, _i64, _int, _p, _i64, _p, _sz, _p]),
    "qgemm_s8_noalloc": (_int, [_i64, _i64, _i64, _p, _i64, _int, _p, _i64, _int, _p, _i64, _p]),
    "qgemm_s8_host": (_int, [_i64, _i64, _i64, _p, _i64, _p, _i64, _p, _i64, _p, _sz, _p]),
    "qgemm_s4": (_int, [_i64, _i64, _i64, _p, _i64, _int, _p, _i64, _int, _p, _i64, _p, _sz, _p]),
    "gemm_f16": (_int, [_i64, _i64, _i64, _p, _i64, _int, _p, _i64, _int, _p, _i64, _p]),
    "w4a16_gemm": (_int, [_i64, _i64, _i64, _p, _i64, _p, _p, _i64, _p, _i64, _p]),
    "w4a4_quantize": (_int, [_i64, _i64, _p, _i64, _p, _i64, _p, _p, _p, _i64, _p]),
    "w4a4_gemm": (_int, [_i64, _i64, _i64, _p, _p, _p, _p, _i64, _p, _p, _i64, _p, _p, _i64,
                         _p, _sz, _p]),
    "w4a4_gemm_affine": (_int, [_i64, _i64, _i64, _p, _p, _p, _p, _i64, _p, _p, _i64, _p, _p, _p,
                                _i64, _p, _sz, _p]),
    "w4a4_prepack_weights": (_int, [_i64, _i64, _p, _p, _i64, _p, _p, _sz, _p]),
    "w4a4_gemm_prepacked": (_int, [_i64, _i64, _i64, _p, _p, _p, _sz, _i64, _p, _p, _i64, _p, _p, _i64,
                                   _p, _sz, _p]),
}

_lib = None


def header_functions() -> list[str]:
    """Names of the functions include/qgemm.h declares."""
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", txt, flags=re.M)


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; "
                f"g.build()\"` (needs nvcc); there is no fallback implementation")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _torch():
    import torch
    return torch


def _stream(stream=None) -> int:
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _check(name: str, code: int) -> None:
    if code != QG_OK:
        err = QgError(name, code)
        if code == 5:  # QG_ERR_CUDA: attach the failing CUDA call's code
            err.cuda_error = int(lib().qg_last_cuda_error())
            err.args = (f"{err.args[0]} (CUDA error code {err.cuda_error})",)
        raise err


def _cuda(t, dtype, name):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() >= 1 and t.stride(-1) != 1:
        raise ValueError(f"{name} must have a contiguous last dimension")
    return t


def workspace_size(op: int, M: int, N: int, K: int) -> int:
    return int(lib().qg_workspace_size(op, M, N, K))


def _workspace(op, M, N, K, device, ws):
    torch = _torch()
    need = workspace_size(op, M, N, K)
    if ws is None:
        # torch's caching allocator returns blocks aligned to at least 512 bytes
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=device)
    return ws, ws.numel() * ws.element_size()


def device_status(stream=None) -> int:
    return int(lib().qg_device_status(_stream(stream)))


STATUS_WORDS = ("code", "site", "count", "block", "parity", "barrier")


def device_status_detail(stream=None) -> dict:
    """Reads and clears the device status word; returns its six fields by name
    ("code" is QG_OK when no wait ran out since the last read)."""
    words = (ctypes.c_int * len(STATUS_WORDS))()
    code = int(lib().qg_device_status_detail(words, _stream(stream)))
    if code == QG_ERR_CUDA:
        raise QgError("qg_device_status_detail", code)
    return dict(zip(STATUS_WORDS, (int(w) for w in words)))


def kernel_budgets(measure: bool = False) -> list:
    """The library's kernel budget table, one dict per kernel instance.  With
    measure=True (needs a device) each entry also gets the compiled kernel's
    registers per thread, static shared memory and the CTAs per SM the
    device's occupancy calculator gives at the entry's launch shape."""
    L = lib()
    out = []
    for i in range(int(L.qg_kernel_budget_count())):
        b = KernelBudgetC()
        _check("qg_kernel_budget_get", L.qg_kernel_budget_get(i, ctypes.byref(b)))
        e = {name: getattr(b, name) for name, _ in KernelBudgetC._fields_}
        e["kernel"] = b.kernel.decode()
        if measure:
            regs, ssm, ctas = _int(), _int(), _int()
            _check("qg_kernel_budget_measure",
                   L.qg_kernel_budget_measure(i, ctypes.byref(regs), ctypes.byref(ssm), ctypes.byref(ctas)))
            e.update(regs_per_thread=regs.value, static_smem_bytes=ssm.value, ctas_per_sm=ctas.value)
        out.append(e)
    return out


def set_timeout_ns(ns: int) -> None:
    _check("qg_set_timeout_ns", lib().qg_set_timeout_ns(int(ns)))


def qgemm_s8(A, B, C=None, ws=None, stream=None):
    torch = _torch()
    _cuda(A, torch.int8, "A")
    _cuda(B, torch.int8, "B")
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K:
        raise ValueError("B must be N x K (K-major)")
    if C is None:
        C = torch.empty((M, N), dtype=torch.int32, device=A.device)
    _cuda(C, torch.int32, "C")
    ws, wsb = _workspace(QG_OP_S8, M, N, K, A.device, ws)
    _check("qgemm_s8", lib().qgemm_s8(M, N, K, A.data_ptr(), A.stride(0), QG_ROW_MAJOR,
                                      B.data_ptr(), B.stride(0), QG_COL_MAJOR,
                                      C.data_ptr(), C.stride(0), ws.data_ptr(), wsb,
                                      _stream(stream)))
    return C


def _host(t, dtype, name):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
        raise TypeError(f"{name} must be a CPU (host) tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != 2 or t.stride(-1) != 1:
        raise ValueError(f"{name} must be a 2-D tensor with unit column stride")


def qgemm_s8_host(A, B, C=None, ws=None, stream=None):
    """qgemm_s8 with A (M x K int8), B (N x K int8) and C (M x N int32) in host
    memory; the copies both ways run inside the call, overlapped with the
    arithmetic.  Use page-locked tensors (``pin_memory()``) for full link
    speed.  The call is asynchronous: C is complete once ``stream`` (default:
    the current stream) has been synchronized.  ``ws`` is a device workspace
    (allocated on the current device when None)."""
    torch = _torch()
    _host(A, torch.int8, "A")
    _host(B, torch.int8, "B")
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K:
        raise ValueError("B must be N x K (K-major)")
    if C is None:
        C = torch.empty((M, N), dtype=torch.int32, pin_memory=A.is_pinned())
    _host(C, torch.int32, "C")
    ws, wsb = _workspace(QG_OP_S8_HOST, M, N, K, torch.device("cuda", torch.cuda.current_device()), ws)
    _check("qgemm_s8_host", lib().qgemm_s8_host(M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0),
                                                C.data_ptr(), C.stride(0), ws.data_ptr(), wsb,
                                                _stream(stream)))
    return C


def qgemm_s4(A, B, K: int, C=None, ws=None, stream=None):
    torch = _torch()
    _cuda(A, torch.uint8, "A")
    _cuda(B, torch.uint8, "B")
    M, N = A.shape[0], B.shape[0]
    if A.shape[1] * 2 < K or B.shape[1] * 2 < K:
        raise ValueError("packed operands must hold K/2 bytes per row")
    if C is None:
        C = torch.empty((M, N), dtype=torch.int32, device=A.device)
    _cuda(C, torch.int32, "C")
    ws, wsb = _workspace(QG_OP_S4, M, N, K, A.device, ws)
    _check("qgemm_s4", lib().qgemm_s4(M, N, K, A.data_ptr(), A.stride(0), QG_ROW_MAJOR,
                                      B.data_ptr(), B.stride(0), QG_COL_MAJOR,
                                      C.data_ptr(), C.stride(0), ws.data_ptr(), wsb,
                                      _stream(stream)))
    return C


def gemm_f16(A, B, C=None, stream=None):
    torch = _torch()
    _cuda(A, torch.float16, "A")
    _cuda(B, torch.float16, "B")
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K:
        raise ValueError("B must be N x K (K-major)")
    if C is None:
        C = torch.empty((M, N), dtype=torch.float16, device=A.device)
    _cuda(C, torch.float16, "C")
    _check("gemm_f16", lib().gemm_f16(M, N, K, A.data_ptr(), A.stride(0), QG_ROW_MAJOR,
                                      B.data_ptr(), B.stride(0), QG_COL_MAJOR,
                                      C.data_ptr(), C.stride(0), _stream(stream)))
    return C


def w4a16_gemm(X, Wq, Wscale, group: int = 128, Y=None, stream=None):
    torch = _torch()
    _cuda(X, torch.float16, "X")
    _cuda(Wq, torch.uint8, "Wq")
    _cuda(Wscale, torch.float16, "Wscale")
    M, K = X.shape
    N = Wq.shape[0]
    if not (Wq.is_contiguous() and Wscale.is_contiguous()):
        raise ValueError("Wq and Wscale must be contiguous")
    if Wq.shape[1] * 2 != K or tuple(Wscale.shape) != (N, K // group):
        raise ValueError("Wq must be N x K/2 bytes and Wscale N x K/group")
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float16, device=X.device)
    _cuda(Y, torch.float16, "Y")
    _check("w4a16_gemm", lib().w4a16_gemm(M, N, K, X.data_ptr(), X.stride(0), Wq.data_ptr(),
                                          Wscale.data_ptr(), group, Y.data_ptr(), Y.stride(0),
                                          _stream(stream)))
    return Y


def w4a4_quantize(X, Ut=None, block: int = 64, out=None, stream=None):
    """Returns (Xq M x K/2 uint8, Xscale M x K/block fp16, XU M x rank fp16 or None).

    Ut is the low-rank down-projection transposed (rank x K fp16, the weight
    of a K -> rank linear layer); XU = X . Ut^T.
    """
    torch = _torch()
    _cuda(X, torch.float32, "X")
    M, K = X.shape
    rank = 0
    U = Ut
    if U is not None:
        _cuda(U, torch.float16, "Ut")
        if not U.is_contiguous() or U.dim() != 2 or U.shape[1] != K:
            raise ValueError("Ut must be a contiguous rank x K fp16 matrix")
        rank = U.shape[0]
    if out is None:
        Xq = torch.empty((M, K // 2), dtype=torch.uint8, device=X.device)
        Xs = torch.empty((M, K // block), dtype=torch.float16, device=X.device)
        XU = torch.empty((M, rank), dtype=torch.float16, device=X.device) if rank else None
    else:
        Xq, Xs, XU = out
    _check("w4a4_quantize", lib().w4a4_quantize(
        M, K, X.data_ptr(), X.stride(0), U.data_ptr() if rank else None, rank,
        Xq.data_ptr(), Xs.data_ptr(), XU.data_ptr() if rank else None, block, _stream(stream)))
    return Xq, Xs, XU


def w4a4_gemm(Xq, Xscale, Wq, Wscale, K: int, XU=None, Vt=None, bias=None, block: int = 64,
              Y=None, ws=None, stream=None, alpha=None):
    """Y = (Q(X).Q(W)^T) (.) scale + XU . Vt^T + bias, fp16 M x N.

    Vt is the low-rank up-projection transposed (N x rank fp16, the weight of
    a rank -> N linear layer).  With alpha (N fp16 column multipliers) the
    call is w4a4_gemm_affine: Y = alpha (.) ((...) (.) scale + XU . Vt^T) + bias.
    """
    torch = _torch()
    V = Vt
    _cuda(Xq, torch.uint8, "Xq")
    _cuda(Wq, torch.uint8, "Wq")
    _cuda(Xscale, torch.float16, "Xscale")
    _cuda(Wscale, torch.float16, "Wscale")
    M, N = Xq.shape[0], Wq.shape[0]
    rank = 0
    if XU is not None:
        _cuda(XU, torch.float16, "XU")
        _cuda(V, torch.float16, "Vt")
        rank = XU.shape[1]
        if not V.is_contiguous() or V.dim() != 2 or V.shape != (N, rank):
            raise ValueError("Vt must be a contiguous N x rank fp16 matrix")
    if bias is not None:
        _cuda(bias, torch.float16, "bias")
    if alpha is not None:
        _cuda(alpha, torch.float16, "alpha")
        if alpha.numel() != N:
            raise ValueError("alpha must hold N fp16 column multipliers")
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float16, device=Xq.device)
    _cuda(Y, torch.float16, "Y")
    ws, wsb = _workspace(QG_OP_W4A4, M, N, K, Xq.device, ws)
    head = (M, N, K, Xq.data_ptr(), Xscale.data_ptr(), Wq.data_ptr(), Wscale.data_ptr(), block,
            XU.data_ptr() if rank else None, V.data_ptr() if rank else None, rank)
    tail = (bias.data_ptr() if bias is not None else None, Y.data_ptr(), Y.stride(0),
            ws.data_ptr(), wsb, _stream(stream))
    if alpha is None:
        _check("w4a4_gemm", lib().w4a4_gemm(*head, *tail))
    else:
        _check("w4a4_gemm_affine", lib().w4a4_gemm_affine(*head, alpha.data_ptr(), *tail))
    return Y


def w4a4_prepack_weights(Wq, Wscale, K: int, alpha=None, block: int = 64, out=None, stream=None):
    """The weight side of w4a4_gemm prepared once: a uint8 device buffer for
    w4a4_gemm_prepacked (with the column multiplier alpha folded in, if given)."""
    torch = _torch()
    _cuda(Wq, torch.uint8, "Wq")
    _cuda(Wscale, torch.float16, "Wscale")
    N = Wq.shape[0]
    if alpha is not None:
        _cuda(alpha, torch.float16, "alpha")
        if alpha.numel() != N:
            raise ValueError("alpha must hold N fp16 column multipliers")
    nbytes = workspace_size(QG_OP_W4A4_WEIGHTS, 1, N, K)
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=Wq.device)
    _check("w4a4_prepack_weights", lib().w4a4_prepack_weights(
        N, K, Wq.data_ptr(), Wscale.data_ptr(), block,
        alpha.data_ptr() if alpha is not None else None, out.data_ptr(), out.numel(), _stream(stream)))
    return out


def w4a4_gemm_prepacked(Xq, Xscale, packed, N: int, K: int, XU=None, Vt=None, bias=None, block: int = 64,
                        Y=None, ws=None, stream=None):
    """w4a4_gemm with weights from w4a4_prepack_weights (only X is converted per call)."""
    torch = _torch()
    _cuda(Xq, torch.uint8, "Xq")
    _cuda(Xscale, torch.float16, "Xscale")
    _cuda(packed, torch.uint8, "packed")
    M = Xq.shape[0]
    rank = 0
    V = Vt
    if XU is not None:
        _cuda(XU, torch.float16, "XU")
        _cuda(V, torch.float16, "Vt")
        rank = XU.shape[1]
        if not V.is_contiguous() or V.dim() != 2 or V.shape != (N, rank):
            raise ValueError("Vt must be a contiguous N x rank fp16 matrix")
    if bias is not None:
        _cuda(bias, torch.float16, "bias")
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float16, device=Xq.device)
    _cuda(Y, torch.float16, "Y")
    ws, wsb = _workspace(QG_OP_W4A4_PREPACKED, M, N, K, Xq.device, ws)
    _check("w4a4_gemm_prepacked", lib().w4a4_gemm_prepacked(
        M, N, K, Xq.data_ptr(), Xscale.data_ptr(), packed.data_ptr(), packed.numel(), block,
        XU.data_ptr() if rank else None, V.data_ptr() if rank else None, rank,
        bias.data_ptr() if bias is not None else None, Y.data_ptr(), Y.stride(0),
        ws.data_ptr(), wsb, _stream(stream)))
    return Y
