"""CPU oracle for the quantized GEMM path (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline may import this package.  The product library never does, and the
product path fails loudly when its CUDA library is missing instead of falling
back to anything here.

The arithmetic lives in ``qgemm_oracle.c`` (plain C, int64 / double
accumulation).  This module compiles it with gcc, loads it with ctypes and
wraps each function for numpy arrays.  Output rows are independent, so large
calls are split over row blocks on a thread pool (ctypes releases the GIL
while the C loop runs); the arithmetic inside a row is untouched.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qgemm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_p = ctypes.c_void_p


CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (gcc, no fast-math)."""
    with _lock:
        if (not force and os.path.exists(_LIB)
                and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
            return _LIB
        tmp = _LIB + ".tmp%d" % os.getpid()
        cmd = ["gcc"] + CFLAGS + [_SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
        return _LIB


def _load():
    global _lib
    if _lib is None:
        # ORACLE_LIB_PATH: a build of a modified copy of the source, loaded
        # instead (the mutation test plants one mistake per build and checks
        # that the pins catch it)
        lib = ctypes.CDLL(os.environ.get("ORACLE_LIB_PATH") or build())
        sig = {
            "orc_half_to_double": (ctypes.c_double, [ctypes.c_uint16]),
            "orc_float_to_half": (ctypes.c_uint16, [ctypes.c_float]),
            "orc_double_to_half": (ctypes.c_uint16, [ctypes.c_double]),
            "orc_s4_unpack": (ctypes.c_int, [_i64, _i64, _p, _i64, _p, _i64]),
            "orc_s4_pack": (ctypes.c_int, [_i64, _i64, _p, _i64, _p, _i64]),
            "orc_gemm_s8": (ctypes.c_int, [_i64, _i64, _i64, _p, _i64, _p, _i64, _p, _i64]),
            "orc_gemm_s4": (ctypes.c_int, [_i64, _i64, _i64, _p, _i64, _p, _i64, _p, _i64]),
            "orc_gemm_f16": (ctypes.c_int, [_i64, _i64, _i64, _p, _i64, _p, _i64, _p, _i64]),
            "orc_w4a16": (ctypes.c_int, [_i64, _i64, _i64, _p, _i64, _p, _i64, _p, _i64,
                                         _i64, _p, _i64]),
            "orc_w4a4_quantize": (ctypes.c_int, [_i64, _i64, _p, _i64, _i64, _p, _i64,
                                                 _p, _i64]),
            "orc_lowrank_xu": (ctypes.c_int, [_i64, _i64, _i64, _p, _i64, _p, _i64,
                                              _p, _i64]),
            "orc_w4a4_gemm": (ctypes.c_int, [_i64, _i64, _i64, _p, _i64, _p, _i64,
                                             _p, _i64, _p, _i64, _i64, _p, _i64,
                                             _p, _i64, _i64, _p, _p, _p, _i64]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def threads() -> int:
    """Worker threads used for row-parallel calls (the host cores we may use)."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _ptr(a: np.ndarray | None) -> int | None:
    return None if a is None else a.ctypes.data


def _check(rc: int, name: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {name} failed with code {rc}")


def _rows_parallel(M: int, fn, nthreads: int | None = None) -> None:
    """Run fn(r0, r1) over row blocks covering [0, M)."""
    n = threads() if nthreads is None else nthreads
    if M <= 1 or n <= 1:
        fn(0, M)
        return
    step = max(1, -(-M // (4 * n)))
    blocks = [(r, min(M, r + step)) for r in range(0, M, step)]
    with ThreadPoolExecutor(max_workers=n) as ex:
        for f in [ex.submit(fn, a, b) for a, b in blocks]:
            f.result()


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


# ---- fp16 conversions ----

def half_to_double(h: int) -> float:
    return _load().orc_half_to_double(int(h) & 0xFFFF)


def float_to_half(x: float) -> int:
    return _load().orc_float_to_half(float(x))


def double_to_half(x: float) -> int:
    return _load().orc_double_to_half(float(x))


def halves_to_double(h: np.ndarray) -> np.ndarray:
    """Elementwise binary16 (uint16 bits) -> double, via the oracle's conversion."""
    h = np.ascontiguousarray(h, dtype=np.uint16)
    f = _load().orc_half_to_double
    return np.array([f(int(v)) for v in h.ravel()], dtype=np.float64).reshape(h.shape)


# ---- 4-bit packing ----

def s4_unpack(P: np.ndarray, K: int) -> np.ndarray:
    P = _c(P, np.uint8)
    rows = P.shape[0]
    V = np.empty((rows, K), dtype=np.int8)
    _check(_load().orc_s4_unpack(rows, K, _ptr(P), P.shape[1], _ptr(V), K), "s4_unpack")
    return V


def s4_pack(V: np.ndarray) -> np.ndarray:
    V = _c(V, np.int8)
    rows, K = V.shape
    P = np.empty((rows, K // 2), dtype=np.uint8)
    _check(_load().orc_s4_pack(rows, K, _ptr(V), K, _ptr(P), K // 2), "s4_pack")
    return P


# ---- GEMMs ----

def gemm_s8(A: np.ndarray, B: np.ndarray, nthreads: int | None = None) -> np.ndarray:
    """C = A . B^T exactly, A: M x K int8, B: N x K int8 (K-major), C int32."""
    A, B = _c(A, np.int8), _c(B, np.int8)
    M, K = A.shape
    N = B.shape[0]
    assert B.shape[1] == K
    C = np.empty((M, N), dtype=np.int32)
    lib = _load()

    def run(r0, r1):
        _check(lib.orc_gemm_s8(r1 - r0, N, K, _ptr(A[r0:r1]), K, _ptr(B), K,
                               _ptr(C[r0:r1]), N), "gemm_s8")
    _rows_parallel(M, run, nthreads)
    return C


def gemm_s4(A: np.ndarray, B: np.ndarray, K: int, nthreads: int | None = None) -> np.ndarray:
    """C = A . B^T exactly on packed s4 operands (M x K/2 and N x K/2 bytes)."""
    A, B = _c(A, np.uint8), _c(B, np.uint8)
    M, N = A.shape[0], B.shape[0]
    assert A.shape[1] == K // 2 and B.shape[1] == K // 2
    C = np.empty((M, N), dtype=np.int32)
    lib = _load()

    def run(r0, r1):
        _check(lib.orc_gemm_s4(r1 - r0, N, K, _ptr(A[r0:r1]), K // 2, _ptr(B), K // 2,
                               _ptr(C[r0:r1]), N), "gemm_s4")
    _rows_parallel(M, run, nthreads)
    return C


def gemm_f16(A: np.ndarray, B: np.ndarray, nthreads: int | None = None) -> np.ndarray:
    """C = A . B^T in double, A: M x K fp16, B: N x K fp16."""
    A = _c(A.view(np.uint16) if A.dtype == np.float16 else A, np.uint16)
    B = _c(B.view(np.uint16) if B.dtype == np.float16 else B, np.uint16)
    M, K = A.shape
    N = B.shape[0]
    C = np.empty((M, N), dtype=np.float64)
    lib = _load()

    def run(r0, r1):
        _check(lib.orc_gemm_f16(r1 - r0, N, K, _ptr(A[r0:r1]), K, _ptr(B), K,
                                _ptr(C[r0:r1]), N), "gemm_f16")
    _rows_parallel(M, run, nthreads)
    return C


def w4a16(X: np.ndarray, Wq: np.ndarray, S: np.ndarray, group: int,
          nthreads: int | None = None) -> np.ndarray:
    """Y = X . (s (.) q)^T in double.  X: M x K fp16, Wq: N x K/2 s4p, S: N x K/group fp16."""
    X = _c(X.view(np.uint16) if X.dtype == np.float16 else X, np.uint16)
    S = _c(S.view(np.uint16) if S.dtype == np.float16 else S, np.uint16)
    Wq = _c(Wq, np.uint8)
    M, K = X.shape
    N = Wq.shape[0]
    Y = np.empty((M, N), dtype=np.float64)
    lib = _load()

    def run(r0, r1):
        _check(lib.orc_w4a16(r1 - r0, N, K, _ptr(X[r0:r1]), K, _ptr(Wq), K // 2,
                             _ptr(S), S.shape[1], group, _ptr(Y[r0:r1]), N), "w4a16")
    _rows_parallel(M, run, nthreads)
    return Y


def w4a4_quantize(X: np.ndarray, block: int, nthreads: int | None = None):
    """Q(X): returns (q packed s4p M x K/2 uint8, scales M x K/block uint16 fp16 bits)."""
    X = _c(X, np.float32)
    M, K = X.shape
    Q = np.empty((M, K // 2), dtype=np.uint8)
    S = np.empty((M, K // block), dtype=np.uint16)
    lib = _load()

    def run(r0, r1):
        _check(lib.orc_w4a4_quantize(r1 - r0, K, _ptr(X[r0:r1]), K, block,
                                     _ptr(Q[r0:r1]), K // 2, _ptr(S[r0:r1]), K // block),
               "w4a4_quantize")
    _rows_parallel(M, run, nthreads)
    return Q, S


def lowrank_xu(X: np.ndarray, U: np.ndarray, nthreads: int | None = None) -> np.ndarray:
    """XU = X . U in double.  X: M x K fp32, U: K x R fp16."""
    X = _c(X, np.float32)
    U = _c(U.view(np.uint16) if U.dtype == np.float16 else U, np.uint16)
    M, K = X.shape
    R = U.shape[1]
    XU = np.empty((M, R), dtype=np.float64)
    lib = _load()

    def run(r0, r1):
        _check(lib.orc_lowrank_xu(r1 - r0, K, R, _ptr(X[r0:r1]), K, _ptr(U), R,
                                  _ptr(XU[r0:r1]), R), "lowrank_xu")
    _rows_parallel(M, run, nthreads)
    return XU


def w4a4_gemm(QX, SX, QW, SW, block: int, K: int, XU=None, V=None, bias=None,
              alpha=None, nthreads: int | None = None) -> np.ndarray:
    """Y = alpha (.) ((Q(X).Q(W)^T) (.) scale + XU.V) + b in double.

    QX: M x K/2 s4p, SX: M x K/block fp16 bits, QW: N x K/2, SW: N x K/block,
    XU: M x R double (or None), V: R x N fp16 (or None), bias: N fp16 (or None),
    alpha: N fp16 column multipliers of the affine calibration (None = 1).
    """
    QX, QW = _c(QX, np.uint8), _c(QW, np.uint8)
    SX = _c(SX.view(np.uint16) if SX.dtype == np.float16 else SX, np.uint16)
    SW = _c(SW.view(np.uint16) if SW.dtype == np.float16 else SW, np.uint16)
    M, N = QX.shape[0], QW.shape[0]
    R = 0
    if XU is not None:
        XU = _c(XU, np.float64)
        V = _c(V.view(np.uint16) if V.dtype == np.float16 else V, np.uint16)
        R = XU.shape[1]
        assert V.shape == (R, N)
    if bias is not None:
        bias = _c(bias.view(np.uint16) if bias.dtype == np.float16 else bias, np.uint16)
        assert bias.shape == (N,)
    if alpha is not None:
        alpha = _c(alpha.view(np.uint16) if alpha.dtype == np.float16 else alpha, np.uint16)
        assert alpha.shape == (N,)
    Y = np.empty((M, N), dtype=np.float64)
    lib = _load()

    def run(r0, r1):
        _check(lib.orc_w4a4_gemm(r1 - r0, N, K, _ptr(QX[r0:r1]), K // 2,
                                 _ptr(SX[r0:r1]), K // block, _ptr(QW), K // 2,
                                 _ptr(SW), K // block, block,
                                 _ptr(XU[r0:r1]) if R else None, R,
                                 _ptr(V) if R else None, N, R,
                                 _ptr(alpha), _ptr(bias), _ptr(Y[r0:r1]), N), "w4a4_gemm")
    _rows_parallel(M, run, nthreads)
    return Y
