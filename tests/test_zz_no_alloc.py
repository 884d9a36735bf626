"""gemm_f32_noalloc: the FP32 entry point for callers that cannot allocate
device memory (code under a fixed device-memory budget, inside an
allocator's callbacks, or where an allocation could block).  Its split
pieces keep their counters and partial sums in a fixed array inside the
library instead of pool memory.

Each case calls it twice in a row (the second call reuses the array the
first left behind) and checks both results against the oracle's D within
the FP32 tolerance of the parity tests.  It must pick gemm_f32's kernel for
the same problem, and take no memory from the library's pool.  A problem
needing more scratch than the array holds is refused before anything is
enqueued.  This file is collected last so that a run stopping at the first
failure has run every other test first.
"""
import numpy as np
import pytest
import torch

import dense_gemm_08_gb300 as lib
from dense_gemm_08_gb300.inputs import COL, ROW, Workload, make_inputs, output_buffer
from gemm_harness import assert_within, c_logical, logical_d, oracle_full

pytestmark = pytest.mark.gpu

CASES = [
    # (workload, expected kernel prefix)
    # last partial wave of 128 x 128 tiles dealt out along K
    (Workload("noalloc_tail", 2560, 2048, 512, 1.5, -0.25, "f32", ROW, ROW, ROW), "sgemm_simt<f32"),
    # fewer tiles than SMs: every tile dealt out along K
    (Workload("noalloc_all_split", 384, 384, 1000, 1.5, -0.25, "f32", ROW, ROW, ROW),
     "sgemm_simt<f32"),
    # M <= 8: the small-M kernel, its K slices added through the array
    (Workload("noalloc_small_m", 4, 3000, 5000, 1.5, -0.25, "f32", ROW, ROW, ROW), "skinny<f32"),
    # column-major D with 6 columns: the call is rewritten as the row-major
    # D^T (6 x 700), which the small-M kernel takes
    (Workload("noalloc_col_d", 700, 6, 3000, 1.0, 0.5, "f32", COL, ROW, COL), "skinny<f32"),
    # a small problem: the cluster kernel (no scratch at all)
    (Workload("noalloc_cluster", 256, 256, 256, 1.0, 0.0, "f32", ROW, ROW, ROW), "sgemm_cluster"),
]


def _call(fn, w, inp, A, B, C, D, ldd):
    return fn(w.M, w.N, w.K, w.alpha, A, inp["lda"], w.order_a, B, inp["ldb"], w.order_b, w.beta,
              C, inp["ldc"], D, ldd, w.order_cd, check=False)


@pytest.mark.parametrize("case", CASES, ids=[w.name for w, _ in CASES])
def test_noalloc_matches_the_oracle_on_two_calls(case):
    w, prefix = case
    inp = make_inputs(w, seed=21)
    A, B = inp["A"].cuda(), inp["B"].cuda()
    C = inp["C"].cuda() if inp["C"] is not None else None
    ref, S = oracle_full(w, inp)
    Cv = c_logical(w, inp)
    # the allocating entry point's choice of kernel for this problem
    Dg, ldd = output_buffer(w, device="cuda", fill=0.0)
    assert _call(lib.gemm_f32, w, inp, A, B, C, Dg, ldd) == lib.GEMM_OK
    want_kernel = lib.gemm_last_kernel()
    assert want_kernel.startswith(prefix), want_kernel
    torch.cuda.synchronize()
    # calls of this entry point take nothing from the library's pool
    assert lib.gemm_release_memory() == lib.GEMM_OK
    for call in range(2):
        D, ldd = output_buffer(w, device="cuda", fill=float("nan"))
        assert _call(lib.gemm_f32_noalloc, w, inp, A, B, C, D, ldd) == lib.GEMM_OK
        assert lib.gemm_last_kernel() == want_kernel
        torch.cuda.synchronize()
        got = logical_d(w, D.cpu())
        assert np.isfinite(got).all(), f"call {call}"
        assert_within(w, got, ref, S, Cv, f"noalloc call {call}")
    info = lib.gemm_memory_info()
    assert info["pool_used_bytes"] == 0 and info["pool_reserved_bytes"] == 0, info
    assert info["split_streams"] == 0, info


def test_noalloc_refuses_a_problem_beyond_its_scratch():
    # One row of 128 x 256 tiles, 3 x SMs - 1 of them, K = 2048 (128 slices of
    # 16): the last SMs - 1 tiles are dealt out along K to all SMs, each tile
    # to at least 2 CTAs, so the partial sums need at least
    # (SMs - 1) x 2 x 128 KiB -- more than the 32 MiB array from 130 SMs on.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms < 130:
        pytest.skip(f"{sms} SMs: this shape fits the array")
    M, N, K = 128, 256 * (3 * sms - 1), 2048
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
    assert lib.gemm_last_kernel().startswith("sgemm_simt<f32")
    torch.cuda.synchronize()
    assert torch.all(D == 0.0)
