"""CPU oracle for D = alpha*op(A)*op(B) + beta*C  -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference arm may import this package.  The CUDA library never
calls it, and it shares no code with the library: the arithmetic lives in
``gemm_oracle.c`` (plain C, double accumulation, POSIX threads), this module
only builds that file with gcc and marshals numpy arrays into it.

The definition it follows is the GEMM definition of "GEMM on NVIDIA GPUs:
from naive kernel to tiled pipeline", section 1: D_ij = alpha * sum_k A_ik
B_kj + beta * C_ij.  ``tiled_counted`` (same package) restates the tiled
counting model of "Understanding roofline and tiling through matrix
multiplication", sections 6.2-6.3 and 10.2, used to pin this oracle.

Storage orders: ``ROW`` stores X(r, q) at X[r*ld + q], ``COL`` at X[r + q*ld].
BF16 operands are passed as their raw 16-bit patterns (numpy uint16), FP16
operands as numpy float16 arrays (read as binary16 bit patterns).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

ROW = 0
COL = 1
IN_F32 = 0
IN_BF16 = 1
IN_F16 = 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_gemm.so")
_lock = threading.Lock()
_lib = None

# -O2, no fast-math, no FMA contraction: the double arithmetic is the
# plain IEEE sequence written in the source, on x86 and on Arm alike.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread"]


def build(force: bool = False) -> str:
    """Compile gemm_oracle.c into liboracle_gemm.so next to it (gcc)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, dbl, vp, ip = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
            lib.oracle_gemm.argtypes = [ip, i64, i64, i64, dbl, vp, i64, ip, vp, i64, ip, dbl,
                                        vp, i64, ip, vp, vp, ip]
            lib.oracle_gemm.restype = ip
            lib.oracle_gemm_points.argtypes = [ip, i64, i64, i64, dbl, vp, i64, ip, vp, i64, ip,
                                               dbl, vp, i64, ip, i64, vp, vp, vp, vp, ip]
            lib.oracle_gemm_points.restype = ip
            lib.oracle_epilogue.argtypes = [i64, i64, vp, vp, ip]
            lib.oracle_epilogue.restype = ip
            lib.oracle_default_threads.argtypes = []
            lib.oracle_default_threads.restype = ip
            _lib = lib
    return _lib


def default_threads() -> int:
    return int(_load().oracle_default_threads())


def _ptr(x):
    if x is None:
        return None
    assert isinstance(x, np.ndarray) and x.flags.c_contiguous
    return x.ctypes.data


def _in_type(a) -> int:
    if a is None:
        return IN_F32
    if a.dtype == np.float32:
        return IN_F32
    if a.dtype == np.uint16:
        return IN_BF16
    if a.dtype == np.float16:
        return IN_F16
    raise TypeError(f"oracle operands are float32, uint16 (bf16 bits) or float16, got {a.dtype}")


def _common(M, N, K, alpha, A, lda, order_a, B, ldb, order_b, beta, C, ldc, order_c):
    ta = _in_type(A)
    tb = _in_type(B)
    if A is not None and B is not None and ta != tb:
        raise TypeError("A and B must have the same element type")
    if C is not None and C.dtype != np.float32:
        raise TypeError("C is float32")
    in_type = ta if A is not None else tb
    return (in_type, int(M), int(N), int(K), float(alpha), _ptr(A), int(lda), int(order_a),
            _ptr(B), int(ldb), int(order_b), float(beta), _ptr(C), int(ldc), int(order_c))


def gemm(M, N, K, alpha, A, lda, order_a, B, ldb, order_b, beta=0.0, C=None, ldc=1,
         order_c=ROW, nthreads=0):
    """Whole result.  Returns (D, S): float64 arrays of shape (M, N).

    D is alpha*sum_k A_ik B_kj + beta*C_ij in double; S is sum_k |alpha A_ik B_kj|.
    Round D to float32 (numpy astype, round-to-nearest-even) for the FP32 value.
    """
    D = np.zeros((M, N), dtype=np.float64)
    S = np.zeros((M, N), dtype=np.float64)
    args = _common(M, N, K, alpha, A, lda, order_a, B, ldb, order_b, beta, C, ldc, order_c)
    rc = _load().oracle_gemm(*args, D.ctypes.data, S.ctypes.data, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gemm rejected its arguments")
    return D, S


def gemm_points(M, N, K, alpha, A, lda, order_a, B, ldb, order_b, beta, C, ldc, order_c, I, J,
                nthreads=0):
    """Selected entries (I[t], J[t]).  Returns (D, S) float64 vectors."""
    I = np.ascontiguousarray(I, dtype=np.int64)
    J = np.ascontiguousarray(J, dtype=np.int64)
    D = np.zeros(I.shape[0], dtype=np.float64)
    S = np.zeros(I.shape[0], dtype=np.float64)
    args = _common(M, N, K, alpha, A, lda, order_a, B, ldb, order_b, beta, C, ldc, order_c)
    rc = _load().oracle_gemm_points(*args, int(I.shape[0]), I.ctypes.data, J.ctypes.data,
                                    D.ctypes.data, S.ctypes.data, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gemm_points rejected its arguments")
    return D, S


ACT_NONE = 0
ACT_RELU = 1
ACT_GELU = 2


def epilogue(D, bias=None, act=ACT_NONE):
    """In place on a float64 (M, N) result: D = act(D + bias[None, :]).

    act: ACT_NONE, ACT_RELU (max(x, 0)) or ACT_GELU (tanh form).  Returns D.
    """
    assert D.dtype == np.float64 and D.flags.c_contiguous and D.ndim == 2
    if bias is not None:
        bias = np.ascontiguousarray(bias, dtype=np.float32)
        assert bias.shape == (D.shape[1],)
    rc = _load().oracle_epilogue(D.shape[0], D.shape[1], D.ctypes.data, _ptr(bias), int(act))
    if rc != 0:
        raise ValueError("oracle_epilogue rejected its arguments")
    return D
