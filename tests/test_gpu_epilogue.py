"""GPU parity of gemm_bf16_f32acc_ex: D = act(alpha*AB + beta*C + bias), FP32 or BF16.

The oracle gives the exact pre-activation value in double, then its own
epilogue; the bound is the BF16 path's 4e-3 * S + 1e-6 on the pre-activation
value, times 1.13 for GELU (its largest slope) plus 1e-6 |y|, and for a BF16
D plus 2^-8 |y|: BF16 keeps 8 significant bits, so rounding to nearest moves
a value by at most half an ulp, 2^-8 of its magnitude.
"""
import itertools

import numpy as np
import pytest
import torch

import dense_gemm_08_gb300 as lib
import oracle
from dense_gemm_08_gb300.inputs import COL, ROW, Workload, make_inputs
from gemm_harness import np_bits, oracle_full

pytestmark = pytest.mark.gpu

ACTS = [lib.GEMM_ACT_NONE, lib.GEMM_ACT_RELU, lib.GEMM_ACT_GELU]
DTYPES = [lib.GEMM_D_F32, lib.GEMM_D_BF16]


def run_ex(w, inp, bias, act, d_type, pad_d=0):
    A = inp["A"].to("cuda")
    B = inp["B"].to("cuda")
    C = inp["C"].to("cuda") if inp["C"] is not None else None
    rows, cols = (w.M, w.N) if w.order_cd == ROW else (w.N, w.M)
    ldd = cols + pad_d
    tdt = torch.float32 if d_type == lib.GEMM_D_F32 else torch.bfloat16
    D = torch.full((max(rows, 1) + 2, ldd), 77.0, dtype=tdt, device="cuda")
    b = torch.from_numpy(bias).to("cuda") if bias is not None else None
    lib.gemm_bf16_f32acc_ex(w.M, w.N, w.K, w.alpha, A, inp["lda"], w.order_a, B, inp["ldb"],
                            w.order_b, w.beta, C, inp["ldc"], D, ldd, w.order_cd, bias=b,
                            activation=act, d_type=d_type)
    name = lib.gemm_last_kernel()
    torch.cuda.synchronize()
    assert lib.gemm_last_device_status() == lib.GEMM_OK
    Dc = D.float().cpu().numpy()
    # guard band: the spare rows and columns still hold 77
    spare = Dc.copy()
    spare[:rows, :cols] = 77.0
    assert np.all(spare == 77.0), "store outside D"
    got = Dc[:rows, :cols] if w.order_cd == ROW else Dc[:rows, :cols].T
    return got, name


def check(w, inp, bias, act, d_type, pad_d=0, expect=None, staged=False):
    got, name = run_ex(w, inp, bias, act, d_type, pad_d)
    if expect:
        assert name.startswith(expect), name
    if staged:
        assert "direct" not in name, name
    x, S = oracle_full(w, inp)  # pre-activation value in double
    y = oracle.epilogue(np.ascontiguousarray(x), bias, act)
    tol = 4e-3 * S + 1e-6
    if act == lib.GEMM_ACT_GELU:
        tol = 1.13 * tol + 1e-6 * np.abs(y)
    if d_type == lib.GEMM_D_BF16:
        tol = tol * (1 + 2.0 ** -8) + 2.0 ** -8 * np.abs(y)
    err = np.abs(got.astype(np.float64) - y)
    bad = ~(err <= tol)
    assert not bad.any(), (f"{int(bad.sum())} entries outside the bound, worst err/tol "
                           f"{np.nanmax(err / np.maximum(tol, 1e-300)):.3g}")


def bias_for(w, seed):
    rng = np.random.default_rng(seed)
    return rng.normal(size=w.N).astype(np.float32)


@pytest.mark.parametrize("act,d_type", list(itertools.product(ACTS, DTYPES)))
@pytest.mark.parametrize("with_bias", [False, True])
def test_epilogue_tensor_core_moderate(act, d_type, with_bias):
    w = Workload("epi", 300, 600, 200, 1.5, -0.25, "bf16", ROW, COL, ROW)
    inp = make_inputs(w, seed=31, ld_multiple=8)
    bias = bias_for(w, 32) if with_bias else None
    check(w, inp, bias, act, d_type, pad_d=8, expect="gemm_bf16_tc")


@pytest.mark.parametrize("variant", ["pair", "pair_staged", "pair_tail", "splitk", "simt",
                                     "scale_c", "col_major_d", "unaligned_d", "ragged_n",
                                     "narrow_n", "small_m"])
@pytest.mark.parametrize("d_type", DTYPES)
def test_epilogue_every_path(variant, d_type):
    shapes = {"pair": (2500, 2600, 136), "pair_staged": (2500, 2600, 136),
              "pair_tail": (2000, 3300, 777), "splitk": (300, 600, 2048), "simt": (150, 270, 101),
              "scale_c": (70, 90, 0), "col_major_d": (300, 600, 200), "unaligned_d": (300, 601, 200),
              "ragged_n": (300, 601, 200),
              # single CTAs: a 64-row B box (N = 48), a 16-row A box (M = 5)
              "narrow_n": (1000, 48, 700), "small_m": (5, 600, 1000)}
    M, N, K = shapes[variant]
    order_cd = COL if variant == "col_major_d" else ROW
    w = Workload("epi_" + variant, M, N, K, 1.5, -0.25, "bf16", ROW, COL, order_cd)
    inp = make_inputs(w, seed=33, ld_multiple=1 if variant == "simt" else 8)
    bias = bias_for(w, 34)
    expect = {"pair": "gemm_bf16_tc<pair,direct", "pair_staged": "gemm_bf16_tc<pair",
              "pair_tail": "gemm_bf16_tc<pair",
              "splitk": "gemm_bf16_tc<splitk,",
              "simt": "sgemm_simt<bf16", "scale_c": "scale_c", "col_major_d": "gemm_bf16_tc",
              "unaligned_d": "gemm_bf16_tc", "ragged_n": "gemm_bf16_tc",
              "narrow_n": "gemm_bf16_tc", "small_m": "gemm_bf16_tc<splitk,x"}[variant]
    # D rows on 32 bytes (the pair kernel's direct epilogue; TMA stores on the
    # single-CTA kernel) except: pair_staged has 16-byte rows (2604, staged
    # boxes and TMA stores), unaligned_d an odd ldd (603), and ragged_n a
    # 16-byte ldd (608) but rows of 601 elements (both take row stores)
    pad_d = {"pair_staged": 4, "unaligned_d": 2, "ragged_n": 7}.get(variant, 8)
    check(w, inp, bias, lib.GEMM_ACT_GELU, d_type, pad_d=pad_d, expect=expect,
          staged=variant == "pair_staged")


def test_epilogue_null_descriptor_equals_plain_call():
    w = Workload("epi_null", 300, 600, 200, 1.5, -0.25, "bf16", ROW, COL, ROW)
    inp = make_inputs(w, seed=35, ld_multiple=8)
    A, B, C = (inp[k].to("cuda") for k in ("A", "B", "C"))
    D1 = torch.empty((w.M, w.N), device="cuda")
    D2 = torch.empty((w.M, w.N), device="cuda")
    lib.gemm_bf16_f32acc(w.M, w.N, w.K, w.alpha, A, inp["lda"], ROW, B, inp["ldb"], COL, w.beta,
                         C, inp["ldc"], D1, w.N, ROW)
    st = lib.library().gemm_bf16_f32acc_ex(w.M, w.N, w.K, w.alpha, A.data_ptr(), inp["lda"], ROW,
                                           B.data_ptr(), inp["ldb"], COL, w.beta, C.data_ptr(),
                                           inp["ldc"], D2.data_ptr(), w.N, ROW, None,
                                           torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert torch.equal(D1, D2)


def test_epilogue_rejects_bad_descriptors():
    D = torch.zeros((8, 8), device="cuda")
    A = torch.zeros((8, 8), dtype=torch.bfloat16, device="cuda")
    for kw in [dict(activation=5), dict(d_type=3), dict(bias=D.data_ptr() + 2)]:
        st = lib.gemm_bf16_f32acc_ex(8, 8, 8, 1.0, A, 8, ROW, A, 8, COL, 0.0, None, 8, D, 8, ROW,
                                     check=False, **kw)
        assert st == lib.GEMM_ERR_INVALID_VALUE, kw
    # a BF16 D only needs 2-byte alignment
    Dh = torch.zeros((8, 9), dtype=torch.bfloat16, device="cuda")
    st = lib.gemm_bf16_f32acc_ex(8, 8, 8, 1.0, A, 8, ROW, A, 8, COL, 0.0, None, 8,
                                 Dh.data_ptr() + 2, 9, ROW, d_type=lib.GEMM_D_BF16, check=False)
    assert st == lib.GEMM_OK


@pytest.mark.parametrize("variant", ["pair", "pair_tail", "col_major_d"])
@pytest.mark.parametrize("d_type", DTYPES)
def test_epilogue_direct_pair_kernel(variant, d_type):
    """beta = 0 with D rows on 32 bytes: the CTA-pair kernel's direct epilogue
    (bias, GELU and the BF16 conversion in registers, D stored from them),
    whole tiles and split tail tiles, ragged N, row- and column-major D.
    (beta != 0 with C rows on 32 bytes is covered by test_epilogue_every_path.)"""
    shapes = {"pair": (2500, 2600, 136), "pair_tail": (2000, 3300, 777),
              "col_major_d": (2600, 2500, 136)}
    M, N, K = shapes[variant]
    order_cd = COL if variant == "col_major_d" else ROW
    w = Workload("epi_direct_" + variant, M, N, K, 1.5, 0.0, "bf16", ROW, COL, order_cd)
    inp = make_inputs(w, seed=36, ld_multiple=8)
    bias = bias_for(w, 37)
    cols = N if order_cd == ROW else M
    per32 = 8 if d_type == lib.GEMM_D_F32 else 16  # elements in 32 bytes
    pad_d = per32 + (-cols) % per32                # ldd on 32 bytes, plus a guard band
    check(w, inp, bias, lib.GEMM_ACT_GELU, d_type, pad_d=pad_d, expect="gemm_bf16_tc<pair,direct")
