"""Shared test plumbing: run the CUDA library and the oracle on the same bits.

Nothing here computes a GEMM: the GPU side calls the C ABI through the
package binding, the reference side calls the oracle.
"""
from __future__ import annotations

import numpy as np
import torch

import dense_gemm_08_gb300 as lib
import oracle
from dense_gemm_08_gb300.inputs import COL, ROW, Workload, make_inputs, output_buffer

F32_REL = 1e-5   # FP32 bound: 1e-5 * S + 1e-6 * |beta C|
F32_C = 1e-6
BF16_REL = 4e-3  # BF16 bound: 4e-3 * S + 1e-6 (also used for FP16 inputs)
BF16_ABS = 1e-6
SENTINEL = 1234.5


def np_bits(t: torch.Tensor) -> np.ndarray:
    """CPU tensor -> contiguous numpy array the oracle reads (bf16 as uint16 bits)."""
    t = t.contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).reshape(-1)
    if t.dtype == torch.float16:
        return t.view(torch.int16).numpy().view(np.float16).reshape(-1)
    return t.numpy().reshape(-1)


def run_gpu(w: Workload, inp, pad_d: int = 0, device="cuda", stream=None, in_place=False):
    """Call the library on GPU copies of `inp`; returns (D storage on CPU, ldd, kernel name)."""
    A = inp["A"].to(device)
    B = inp["B"].to(device)
    C = inp["C"].to(device) if inp["C"] is not None else None
    if in_place:
        assert C is not None
        Dbuf, ldd = C, inp["ldc"]
    else:
        Dbuf, ldd = output_buffer(w, pad=pad_d, device=device, fill=SENTINEL,
                                  pad_rows=3 if pad_d else 0)
    fn = {"f32": lib.gemm_f32, "bf16": lib.gemm_bf16_f32acc, "f16": lib.gemm_f16_f32acc}[w.dtype]
    fn(w.M, w.N, w.K, w.alpha, A, inp["lda"], w.order_a, B, inp["ldb"], w.order_b, w.beta, C,
       inp["ldc"], Dbuf, ldd, w.order_cd, stream)
    name = lib.gemm_last_kernel()
    torch.cuda.synchronize()
    st = lib.gemm_last_device_status()
    assert st == lib.GEMM_OK, f"device status {st}"
    return Dbuf.cpu(), ldd, name


def logical_d(w: Workload, Dbuf: torch.Tensor) -> np.ndarray:
    """M x N view of D's storage."""
    if w.order_cd == ROW:
        return Dbuf[: w.M, : w.N].numpy()
    return Dbuf[: w.N, : w.M].t().numpy()


def oracle_args(w: Workload, inp):
    C = np_bits(inp["C"]) if inp["C"] is not None else None
    return (w.M, w.N, w.K, w.alpha, np_bits(inp["A"]), inp["lda"], w.order_a, np_bits(inp["B"]),
            inp["ldb"], w.order_b, w.beta, C, inp["ldc"], w.order_cd)


def oracle_full(w: Workload, inp):
    M, N, K, al, A, lda, oa, B, ldb, ob, be, C, ldc, oc = oracle_args(w, inp)
    return oracle.gemm(M, N, K, al, A, lda, oa, B, ldb, ob, be, C, ldc, oc)


def oracle_points(w: Workload, inp, I, J):
    return oracle.gemm_points(*oracle_args(w, inp), I, J)


def c_logical(w: Workload, inp) -> np.ndarray | None:
    return inp["C_logical"].numpy() if inp["C_logical"] is not None else None


def bound(w: Workload, S: np.ndarray, Cvals: np.ndarray | None) -> np.ndarray:
    if w.dtype == "f32":
        b = F32_REL * S
        if w.beta != 0 and Cvals is not None:
            b = b + F32_C * np.abs(w.beta * Cvals.astype(np.float64))
        return b
    return BF16_REL * S + BF16_ABS


def assert_within(w: Workload, got: np.ndarray, ref64: np.ndarray, S: np.ndarray,
                  Cvals: np.ndarray | None, what: str = ""):
    """Element-wise |D - D_ref| <= bound, D_ref = oracle result rounded to FP32."""
    ref = ref64.astype(np.float32).astype(np.float64)
    got = got.astype(np.float64)
    err = np.abs(got - ref)
    tol = bound(w, S, Cvals)
    bad = ~(err <= tol)  # NaN counts as bad
    if bad.any():
        idx = np.argwhere(bad)[:5]
        ratio = np.nanmax(err / np.maximum(tol, 1e-300))
        raise AssertionError(f"{w.name} {what}: {int(bad.sum())} of {bad.size} entries outside "
                             f"the bound, worst err/tol {ratio:.3g}, first at {idx.tolist()}")
    return float(np.max(err / np.maximum(tol, 1e-300))) if err.size else 0.0


def sample_points(M: int, N: int, rng: np.random.Generator, n_random: int = 4000,
                  full_rows=(), full_cols=()):
    """Corners, tile boundaries, whole rows/columns and random entries."""
    I, J = [], []
    for r in full_rows:
        if 0 <= r < M:
            I.extend([r] * N)
            J.extend(range(N))
    for c in full_cols:
        if 0 <= c < N:
            I.extend(range(M))
            J.extend([c] * M)
    edges_m = sorted({x for b in (0, 127, 128, 255, 256, M - 129, M - 128, M - 1) for x in (b,)
                      if 0 <= x < M})
    edges_n = sorted({x for b in (0, 127, 128, 255, 256, 257, N - 257, N - 256, N - 1)
                      for x in (b,) if 0 <= x < N})
    for r in edges_m:
        for c in edges_n:
            I.append(r)
            J.append(c)
    I.extend(rng.integers(0, M, n_random).tolist())
    J.extend(rng.integers(0, N, n_random).tolist())
    return np.array(I, dtype=np.int64), np.array(J, dtype=np.int64)


def check_canary(w: Workload, Dbuf: torch.Tensor):
    """Everything in D's storage outside the M x N matrix still holds the sentinel."""
    buf = Dbuf.numpy().copy()
    if w.order_cd == ROW:
        buf[: w.M, : w.N] = SENTINEL
    else:
        buf[: w.N, : w.M] = SENTINEL
    assert np.all(buf == SENTINEL), f"{w.name}: store outside D"
