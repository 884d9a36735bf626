"""Python binding of the GB300 GEMM library's C ABI (include/gemm.h and
include/gemm_probe.h).

Argument marshalling only: every function here forwards to the in-tree
CUDA library ``libdense_gemm_08_gb300.so``; all arithmetic runs in its
kernels.  Importing this package without the built library raises at the
first call (there is no CPU fallback).

Same names as the C ABI:
    gemm_f32, gemm_bf16_f32acc, gemm_f16_f32acc, gemm_bf16_f32acc_ex,
    gemm_f32_noalloc, gemm_status_string, gemm_last_device_status, gemm_last_kernel,
    gemm_memory_info, gemm_release_memory,
    gemm_probe_tc_bf16, gemm_probe_fma_f32, gemm_probe_wait_timeout
Pointer arguments take an integer device address or a torch CUDA tensor;
``stream`` takes an integer ``cudaStream_t``, a ``torch.cuda.Stream`` or None
(torch's current stream).  A non-zero status raises ``GemmError``.

``gemm(...)`` is a convenience wrapper for torch tensors that reads each
operand's storage order and leading dimension from its strides.
"""
from __future__ import annotations

import ctypes
import os
import threading

ROW_MAJOR = 0
COL_MAJOR = 1

GEMM_OK = 0
GEMM_ERR_INVALID_VALUE = 1
GEMM_ERR_UNSUPPORTED_DEVICE = 2
GEMM_ERR_LAUNCH = 3
GEMM_ERR_TIMEOUT = 4
GEMM_ERR_INTERNAL = 5

# DENSE_GEMM_08_GB300_LIB names another build of the same library (for
# example a variant from _build.build_variant); by default the in-tree build.
LIB_PATH = os.environ.get("DENSE_GEMM_08_GB300_LIB") or os.path.join(
    os.path.dirname(os.path.abspath(__file__)), "libdense_gemm_08_gb300.so")
EXPORTED = ("gemm_f32", "gemm_bf16_f32acc", "gemm_f16_f32acc", "gemm_bf16_f32acc_ex",
            "gemm_f32_noalloc", "gemm_status_string", "gemm_last_device_status",
            "gemm_last_kernel", "gemm_memory_info", "gemm_release_memory",
            "gemm_probe_tc_bf16", "gemm_probe_fma_f32", "gemm_probe_wait_timeout")

GEMM_ACT_NONE = 0
GEMM_ACT_RELU = 1
GEMM_ACT_GELU = 2
GEMM_D_F32 = 0
GEMM_D_BF16 = 1


class MemoryInfo(ctypes.Structure):
    """gemm_memory_info_t: what the library holds on the current device."""
    _fields_ = [("split_streams", ctypes.c_uint64), ("split_bytes", ctypes.c_uint64),
                ("pool_used_bytes", ctypes.c_uint64), ("pool_reserved_bytes", ctypes.c_uint64)]


class Epilogue(ctypes.Structure):
    """gemm_epilogue_t: bias (device pointer or None), activation, d_type."""
    _fields_ = [("bias", ctypes.c_void_p), ("activation", ctypes.c_int), ("d_type", ctypes.c_int)]

_lock = threading.Lock()
_lib = None


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: status {status} ({gemm_status_string(status)})")
        self.status = status


def library() -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"CUDA library {LIB_PATH} is not built; run __graft_entry__.build() "
                    "(or python dense_gemm_08_gb300/_build.py)")
            lib = ctypes.CDLL(LIB_PATH)
            i64, f32, vp, ip = ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int
            sig = [i64, i64, i64, f32, vp, i64, ip, vp, i64, ip, f32, vp, i64, vp, i64, ip, vp]
            lib.gemm_f32.argtypes = sig
            lib.gemm_f32.restype = ip
            lib.gemm_bf16_f32acc.argtypes = sig
            lib.gemm_bf16_f32acc.restype = ip
            lib.gemm_f16_f32acc.argtypes = sig
            lib.gemm_f16_f32acc.restype = ip
            lib.gemm_bf16_f32acc_ex.argtypes = sig[:-1] + [ctypes.POINTER(Epilogue), vp]
            lib.gemm_bf16_f32acc_ex.restype = ip
            lib.gemm_f32_noalloc.argtypes = sig
            lib.gemm_f32_noalloc.restype = ip
            lib.gemm_status_string.argtypes = [ip]
            lib.gemm_status_string.restype = ctypes.c_char_p
            lib.gemm_last_device_status.argtypes = [vp]
            lib.gemm_last_device_status.restype = ip
            lib.gemm_last_kernel.argtypes = []
            lib.gemm_last_kernel.restype = ctypes.c_char_p
            lib.gemm_memory_info.argtypes = [ctypes.POINTER(MemoryInfo)]
            lib.gemm_memory_info.restype = ip
            lib.gemm_release_memory.argtypes = []
            lib.gemm_release_memory.restype = ip
            dp = ctypes.POINTER(ctypes.c_double)
            lib.gemm_probe_tc_bf16.argtypes = [ip, i64, dp, vp]
            lib.gemm_probe_tc_bf16.restype = ip
            lib.gemm_probe_fma_f32.argtypes = [i64, dp, vp]
            lib.gemm_probe_fma_f32.restype = ip
            lib.gemm_probe_wait_timeout.argtypes = [ctypes.c_uint64, vp]
            lib.gemm_probe_wait_timeout.restype = ip
            _lib = lib
    return _lib


def _addr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()  # torch tensor


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream  # torch.cuda.Stream


def _call(fn_name, M, N, K, alpha, A, lda, order_a, B, ldb, order_b, beta, C, ldc, D, ldd,
          order_cd, stream, check):
    fn = getattr(library(), fn_name)
    st = fn(int(M), int(N), int(K), float(alpha), _addr(A), int(lda), int(order_a), _addr(B),
            int(ldb), int(order_b), float(beta), _addr(C), int(ldc), _addr(D), int(ldd),
            int(order_cd), _stream(stream))
    if check and st != GEMM_OK:
        raise GemmError(st, fn_name)
    return st


def gemm_f32(M, N, K, alpha, A, lda, order_a, B, ldb, order_b, beta, C, ldc, D, ldd, order_cd,
             stream=None, check=True) -> int:
    """FP32 GEMM on the CUDA cores (see include/gemm.h)."""
    return _call("gemm_f32", M, N, K, alpha, A, lda, order_a, B, ldb, order_b, beta, C, ldc, D,
                 ldd, order_cd, stream, check)


def gemm_bf16_f32acc(M, N, K, alpha, A, lda, order_a, B, ldb, order_b, beta, C, ldc, D, ldd,
                     order_cd, stream=None, check=True) -> int:
    """BF16-input, FP32-accumulate GEMM (tensor cores when TMA applies; see include/gemm.h)."""
    return _call("gemm_bf16_f32acc", M, N, K, alpha, A, lda, order_a, B, ldb, order_b, beta, C,
                 ldc, D, ldd, order_cd, stream, check)


def gemm_f16_f32acc(M, N, K, alpha, A, lda, order_a, B, ldb, order_b, beta, C, ldc, D, ldd,
                    order_cd, stream=None, check=True) -> int:
    """FP16-input, FP32-accumulate GEMM (same kernels as gemm_bf16_f32acc)."""
    return _call("gemm_f16_f32acc", M, N, K, alpha, A, lda, order_a, B, ldb, order_b, beta, C,
                 ldc, D, ldd, order_cd, stream, check)


def gemm_bf16_f32acc_ex(M, N, K, alpha, A, lda, order_a, B, ldb, order_b, beta, C, ldc, D, ldd,
                        order_cd, bias=None, activation=GEMM_ACT_NONE, d_type=GEMM_D_F32,
                        stream=None, check=True) -> int:
    """gemm_bf16_f32acc with a fused epilogue: D = act(alpha*AB + beta*C + bias), FP32 or BF16."""
    ep = Epilogue(_addr(bias), int(activation), int(d_type))
    st = library().gemm_bf16_f32acc_ex(
        int(M), int(N), int(K), float(alpha), _addr(A), int(lda), int(order_a), _addr(B),
        int(ldb), int(order_b), float(beta), _addr(C), int(ldc), _addr(D), int(ldd),
        int(order_cd), ctypes.byref(ep), _stream(stream))
    if check and st != GEMM_OK:
        raise GemmError(st, "gemm_bf16_f32acc_ex")
    return st


def gemm_f32_noalloc(M, N, K, alpha, A, lda, order_a, B, ldb, order_b, beta, C, ldc, D, ldd,
                     order_cd, stream=None, check=True) -> int:
    """gemm_f32 that allocates nothing: its split-K scratch is a fixed 32 MiB
    array inside the library (for callers that cannot allocate device memory;
    see include/gemm.h for the limits)."""
    return _call("gemm_f32_noalloc", M, N, K, alpha, A, lda, order_a, B, ldb, order_b, beta, C,
                 ldc, D, ldd, order_cd, stream, check)


def gemm_status_string(status: int) -> str:
    return library().gemm_status_string(int(status)).decode()


def gemm_last_device_status(stream=None) -> int:
    return int(library().gemm_last_device_status(_stream(stream)))


def gemm_last_kernel() -> str:
    return library().gemm_last_kernel().decode()


def gemm_memory_info(check=True) -> dict:
    """What the library holds on the current device between calls (see include/gemm.h)."""
    info = MemoryInfo()
    st = library().gemm_memory_info(ctypes.byref(info))
    if check and st != GEMM_OK:
        raise GemmError(st, "gemm_memory_info")
    return {name: int(getattr(info, name)) for name, _ in MemoryInfo._fields_}


def gemm_release_memory(check=True) -> int:
    """Synchronise the device, free every stream's split counters and trim the pool."""
    st = int(library().gemm_release_memory())
    if check and st != GEMM_OK:
        raise GemmError(st, "gemm_release_memory")
    return st


def gemm_probe_tc_bf16(cta_group, n_mma, stream=None, check=True):
    """Enqueue the tensor-pipe probe; returns (status, FLOPs of the launch)."""
    flops = ctypes.c_double(0.0)
    st = library().gemm_probe_tc_bf16(int(cta_group), int(n_mma), ctypes.byref(flops),
                                      _stream(stream))
    if check and st != GEMM_OK:
        raise GemmError(st, "gemm_probe_tc_bf16")
    return st, flops.value


def gemm_probe_fma_f32(trips, stream=None, check=True):
    """Enqueue the FP32 FMA probe; returns (status, FLOPs of the launch)."""
    flops = ctypes.c_double(0.0)
    st = library().gemm_probe_fma_f32(int(trips), ctypes.byref(flops), _stream(stream))
    if check and st != GEMM_OK:
        raise GemmError(st, "gemm_probe_fma_f32")
    return st, flops.value


def gemm_probe_wait_timeout(timeout_ns, stream=None, check=True):
    """Enqueue the bounded-wait probe (a wait that runs out after timeout_ns)."""
    st = library().gemm_probe_wait_timeout(int(timeout_ns), _stream(stream))
    if check and st != GEMM_OK:
        raise GemmError(st, "gemm_probe_wait_timeout")
    return st


# ------------------------------------------------------------ torch helper
def storage_order(t):
    """(order, ld) of a 2-D tensor, from its strides; raises if neither dense-row nor dense-column."""
    if t.dim() != 2:
        raise ValueError("expected a 2-D tensor")
    r, q = t.shape
    s0, s1 = t.stride()
    if s1 == 1 and (s0 >= max(q, 1) or r <= 1):
        return ROW_MAJOR, max(s0, q, 1)
    if s0 == 1 and (s1 >= max(r, 1) or q <= 1):
        return COL_MAJOR, max(s1, r, 1)
    raise ValueError(f"tensor with strides {t.stride()} is neither row- nor column-major")


def gemm(A, B, C=None, alpha=1.0, beta=0.0, out=None, stream=None):
    """D = alpha * A @ B + beta * C for torch CUDA tensors.

    A (M x K) and B (K x N) are float32 (-> gemm_f32), bfloat16
    (-> gemm_bf16_f32acc) or float16 (-> gemm_f16_f32acc); C and the result
    are float32 and share one order
    (``out``'s if given, else C's, else row-major).  Any row- or
    column-major view works (e.g. ``B.t()`` of a contiguous N x K tensor).
    """
    import torch
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError("inner dimensions differ")
    if A.dtype != B.dtype:
        raise TypeError("A and B must share a dtype")
    oa, lda = storage_order(A)
    ob, ldb = storage_order(B)
    if out is None:
        if C is not None and C.shape == (M, N):
            ocd_pref = storage_order(C)[0]
        else:
            ocd_pref = ROW_MAJOR
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
        if ocd_pref == COL_MAJOR:
            out = torch.empty((N, M), dtype=torch.float32, device=A.device).t()
    ocd, ldd = storage_order(out)
    ldc = ldd
    if beta != 0.0:
        if C is None:
            raise ValueError("beta != 0 needs C")
        oc, ldc = storage_order(C)
        if oc != ocd:
            raise ValueError("C and the output must share a storage order")
    fns = {torch.float32: gemm_f32, torch.bfloat16: gemm_bf16_f32acc,
           torch.float16: gemm_f16_f32acc}
    if A.dtype not in fns:
        raise TypeError("A and B must be float32, bfloat16 or float16")
    fn = fns[A.dtype]
    fn(M, N, K, alpha, A, lda, oa, B, ldb, ob, beta, C if beta != 0.0 else None, ldc, out, ldd,
       ocd, stream)
    return out
