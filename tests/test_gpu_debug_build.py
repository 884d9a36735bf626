"""The tensor-core kernel's debug build against the oracle.

`-DGEMM_TC_DEBUG=1` runs every operand ring at its smallest depth (2
stages) and launches one work item per CTA or CTA pair instead of the
persistent grid.  A wrong result in the normal build that this build gets
right points at the ring, its phases or the persistent schedule rather than
at the arithmetic.  The build is a second copy of the library
(`_build.build_variant`), so the checks run in a child process that loads
it; each variant of the kernel is reached: CTA pairs with the direct and
the staged epilogue, a split last round, the single-CTA kernel with the
cluster split-K, narrow-N and small-M tiles.  Results must stay within the
parity tolerance and be bit-exact on small integers.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))

CHILD = r"""
import sys
import numpy as np
import dense_gemm_08_gb300 as lib
from dense_gemm_08_gb300.inputs import COL, ROW, Workload, make_inputs
from gemm_harness import assert_within, c_logical, check_canary, logical_d, oracle_full, run_gpu

assert lib.LIB_PATH.endswith("tc_debug/libdense_gemm_08_gb300.so"), lib.LIB_PATH
cases = [
    # (name, M, N, K, dist, pad_d, expected kernel prefix)
    ("pair_direct", 2500, 2600, 136, "normal", 0, "gemm_bf16_tc<pair,direct"),
    ("pair_staged", 2500, 2600, 136, "normal", 3, "gemm_bf16_tc<pair"),
    ("pair_split_tail", 2304, 2560, 1024, "normal", 0, "gemm_bf16_tc<pair"),
    ("cluster_split", 300, 600, 2048, "normal", 3, "gemm_bf16_tc<splitk,x"),
    ("narrow_n", 1000, 64, 777, "normal", 0, "gemm_bf16_tc"),
    ("small_m", 7, 600, 1000, "normal", 0, "gemm_bf16_tc<splitk,x"),
    ("single_cta_int", 1000, 1000, 640, "int", 0, "gemm_bf16_tc"),
]
for name, M, N, K, dist, pad_d, prefix in cases:
    w = Workload("dbg_" + name, M, N, K, 1.0 if dist == "int" else 1.5,
                 0.0 if dist == "int" else -0.25, "bf16", ROW, COL, ROW, dist=dist)
    inp = make_inputs(w, seed=M + N + K, ld_multiple=8)
    Dbuf, ldd, kname = run_gpu(w, inp, pad_d=pad_d)
    assert kname.startswith(prefix), (name, kname)
    D = logical_d(w, Dbuf)
    ref, S = oracle_full(w, inp)
    if dist == "int":
        assert np.array_equal(D, ref.astype(np.float32)), name
    else:
        assert_within(w, D, ref, S, c_logical(w, inp), name)
    if pad_d:
        check_canary(w, Dbuf)
    print(name, kname, "ok", flush=True)
"""


def test_debug_build_matches_the_oracle():
    from dense_gemm_08_gb300 import _build
    lib_path = _build.build_variant("tc_debug", {"GEMM_TC_DEBUG": 1})
    env = dict(os.environ, DENSE_GEMM_08_GB300_LIB=lib_path)
    env["PYTHONPATH"] = os.pathsep.join([HERE, os.path.dirname(HERE), env.get("PYTHONPATH", "")])
    r = subprocess.run([sys.executable, "-c", CHILD], env=env, cwd=HERE, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert r.stdout.count(" ok") == 7, r.stdout
