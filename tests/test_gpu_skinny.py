"""GPU parity of the small-M kernel (M <= 8 after the column-major D
normalisation): every input type, both layouts of op(A) and op(B), one and
several K slices, wide and scalar loads, ragged N and K, the fused epilogue,
determinism and exactness on small integers.

FP32 problems with M <= 8 always take this kernel; BF16 and FP16 ones take it
when the tensor-core kernel cannot (operands TMA cannot describe), so the
16-bit cases here give A an odd leading dimension and keep B aligned (wide
loads) unless a test asks for scalar loads."""
import itertools

import numpy as np
import pytest
import torch

import dense_gemm_08_gb300 as lib
import oracle
from dense_gemm_08_gb300.inputs import COL, ROW, Workload, _lay_out, make_inputs
from gemm_harness import (assert_within, c_logical, check_canary, logical_d, oracle_full,
                          run_gpu)

pytestmark = pytest.mark.gpu

ORDERS = list(itertools.product((ROW, COL), repeat=3))
# (M, N, K): one K chunk and several (ragged), N ragged against the column
# blocks of both kernels
# (one column block shared by many CTAs; many column blocks of one K chunk)
SHAPES = [(1, 1, 1), (1, 4096, 4096), (2, 130, 7), (3, 1000, 1025), (4, 33, 3000), (5, 257, 256),
          (7, 129, 513), (8, 300, 2049), (1, 16, 100000), (2, 70000, 64)]


def skinny_inputs(w, seed, odd_b=False):
    """Inputs with 16-byte multiple leading dimensions, except: for 16-bit
    types A's is odd (the tensor-core kernel cannot read it), and with odd_b
    B's too (scalar loads of B)."""
    inp = make_inputs(w, seed=seed, ld_multiple=8)

    def odd(x, order):  # the smallest odd leading dimension
        cols = x.shape[1] if order == ROW else x.shape[0]
        return _lay_out(x, order, 1 if cols % 2 == 0 else 2)

    if w.dtype != "f32":
        inp["A"], inp["lda"] = odd(inp["A_logical"], w.order_a)
    if odd_b:
        inp["B"], inp["ldb"] = odd(inp["B_logical"], w.order_b)
    return inp


def check(w, inp, pad_d=3):
    Dbuf, _, name = run_gpu(w, inp, pad_d=pad_d)
    assert name.startswith("skinny<"), name
    ref, S = oracle_full(w, inp)
    assert_within(w, logical_d(w, Dbuf), ref, S, c_logical(w, inp), str((w.M, w.N, w.K)))
    check_canary(w, Dbuf)
    return Dbuf


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("orders", [(ROW, ROW, ROW), (ROW, COL, ROW), (COL, ROW, ROW),
                                    (COL, COL, ROW)])
def test_small_m_shapes_full(dtype, orders):
    for M, N, K in SHAPES:
        w = Workload("skinny", M, N, K, 1.5, -0.25, dtype, *orders)
        check(w, skinny_inputs(w, seed=M * 7 + K))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_column_major_d_with_few_columns(dtype):
    # D column-major with N <= 8: the stored problem is D^T with 8 or fewer rows
    for orders in [o for o in ORDERS if o[2] == COL]:
        for M, N, K in [(1000, 3, 777), (64, 8, 4096), (5, 1, 300)]:
            w = Workload("skinny_t", M, N, K, 0.5, 1.0, dtype, *orders)
            inp = make_inputs(w, seed=N * 11 + K, pad=1)  # odd: not the tensor-core kernel
            check(w, inp, pad_d=1)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_unaligned_leading_dimensions_take_scalar_loads(dtype):
    for orders in [(ROW, ROW, ROW), (ROW, COL, ROW)]:
        w = Workload("skinny_unal", 3, 517, 1001, 1.5, -0.25, dtype, *orders)
        check(w, skinny_inputs(w, seed=29, odd_b=True), pad_d=1)


def test_several_slices_are_deterministic_and_exact_on_integers():
    w = Workload("skinny_int", 6, 2000, 5000, 1.0, 0.0, "bf16", ROW, COL, ROW, dist="int")
    inp = skinny_inputs(w, seed=30)
    D1, _, name = run_gpu(w, inp)
    assert name.startswith("skinny<")
    ref, _ = oracle_full(w, inp)
    assert np.array_equal(logical_d(w, D1), ref.astype(np.float32))
    w = w.with_(dist="normal", alpha=0.5, beta=1.0, dtype="f32", order_b=ROW)
    inp = make_inputs(w, seed=31)
    D1, _, _ = run_gpu(w, inp)
    D2, _, _ = run_gpu(w, inp)
    assert torch.equal(D1, D2)


@pytest.mark.parametrize("act", [lib.GEMM_ACT_NONE, lib.GEMM_ACT_RELU, lib.GEMM_ACT_GELU])
@pytest.mark.parametrize("d_type", [lib.GEMM_D_F32, lib.GEMM_D_BF16])
def test_fused_epilogue(act, d_type):
    w = Workload("skinny_epi", 4, 700, 1500, 1.5, -0.25, "bf16", ROW, COL, ROW)
    inp = skinny_inputs(w, seed=32)
    bias = np.random.default_rng(33).normal(size=w.N).astype(np.float32)
    A, B, C = (inp[k].cuda() for k in ("A", "B", "C"))
    tdt = torch.float32 if d_type == lib.GEMM_D_F32 else torch.bfloat16
    D = torch.full((w.M + 2, w.N + 8), 77.0, dtype=tdt, device="cuda")
    lib.gemm_bf16_f32acc_ex(w.M, w.N, w.K, w.alpha, A, inp["lda"], ROW, B, inp["ldb"], COL,
                            w.beta, C, inp["ldc"], D, w.N + 8, ROW,
                            bias=torch.from_numpy(bias).cuda(), activation=act, d_type=d_type)
    assert lib.gemm_last_kernel().startswith("skinny<bf16")
    # the same problem with aligned operands takes the tensor-core kernel
    assert inp["lda"] % 8 != 0
    torch.cuda.synchronize()
    Dc = D.float().cpu().numpy()
    spare = Dc.copy()
    spare[:w.M, :w.N] = 77.0
    assert np.all(spare == 77.0), "store outside D"
    x, S = oracle_full(w, inp)
    y = oracle.epilogue(np.ascontiguousarray(x), bias, act)
    tol = 4e-3 * S + 1e-6
    if act == lib.GEMM_ACT_GELU:
        tol = 1.13 * tol + 1e-6 * np.abs(y)
    if d_type == lib.GEMM_D_BF16:
        tol = tol * (1 + 2.0 ** -8) + 2.0 ** -8 * np.abs(y)
    assert np.all(np.abs(Dc[:w.M, :w.N] - y) <= tol)
