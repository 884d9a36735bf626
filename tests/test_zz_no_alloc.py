"""gemm_f32_noalloc: the FP32 entry point for callers that cannot allocate
device memory (its split-K partial sums live in a fixed array inside the
library instead of pool memory).

Checked against gemm_f32 on the same inputs, on two calls in a row (the
second reuses the array the first left behind), within the FP32 tolerance of
the parity tests; a problem needing more scratch than the array holds is
refused before anything is enqueued.  This file is collected last so that a
run stopping at the first failure has run every other test first.
"""
import numpy as np
import pytest
import torch

import dense_gemm_08_gb300 as lib
from dense_gemm_08_gb300.inputs import ROW, Workload, make_inputs
from gemm_harness import assert_within, c_logical, oracle_full

pytestmark = pytest.mark.gpu


def _call(fn, w, A, B, C, inp, D):
    return fn(w.M, w.N, w.K, w.alpha, A, inp["lda"], w.order_a, B, inp["ldb"], w.order_b, w.beta,
              C, inp["ldc"], D, w.N, w.order_cd, check=False)


@pytest.mark.parametrize("shape", [(2560, 2048, 512), (384, 384, 1000)])
def test_noalloc_matches_gemm_f32_on_two_calls(shape):
    # both shapes split tiles along K: a last partial wave / every tile
    M, N, K = shape
    w = Workload("noalloc", M, N, K, 1.5, -0.25, "f32", ROW, ROW, ROW)
    inp = make_inputs(w, seed=21)
    A, B, C = (inp[k].to("cuda") for k in ("A", "B", "C"))
    ref_d = torch.empty((M, N), device="cuda")
    assert _call(lib.gemm_f32, w, A, B, C, inp, ref_d) == lib.GEMM_OK
    torch.cuda.synchronize()
    want = ref_d.cpu().numpy()
    _, S = oracle_full(w, inp)  # tolerance scale sum_k |alpha A_ik B_kj|
    Cv = c_logical(w, inp)
    for call in range(2):
        D = torch.full((M, N), float("nan"), device="cuda")
        assert _call(lib.gemm_f32_noalloc, w, A, B, C, inp, D) == lib.GEMM_OK
        assert lib.gemm_last_kernel().startswith("sgemm_simt<f32")
        torch.cuda.synchronize()
        got = D.cpu().numpy()
        assert np.isfinite(got).all(), f"call {call}"
        assert_within(w, got, want.astype(np.float64), S, Cv, f"noalloc call {call}")


def test_noalloc_refuses_a_problem_beyond_its_scratch():
    # 3 x 101 tiles of 128 x 256 on a 152-SM GB300: 151 tiles are dealt out
    # along K, needing about 57 MiB of partial sums -- more than the 32 MiB array
    M, N, K = 384, 25856, 1024
    A = torch.zeros((M, K), device="cuda")
    B = torch.zeros((K, N), device="cuda")
    D = torch.full((M, N), 3.0, device="cuda")
    st = lib.gemm_f32_noalloc(M, N, K, 1.0, A, K, ROW, B, N, ROW, 0.0, None, N, D, N, ROW,
                              check=False)
    assert st == lib.GEMM_ERR_INVALID_VALUE
    assert lib.gemm_last_kernel() == ""
    torch.cuda.synchronize()
    assert torch.all(D == 3.0)
    # the allocating entry point takes the same problem
    assert lib.gemm_f32(M, N, K, 1.0, A, K, ROW, B, N, ROW, 0.0, None, N, D, N, ROW) == 0
    torch.cuda.synchronize()
    assert torch.all(D == 0.0)
