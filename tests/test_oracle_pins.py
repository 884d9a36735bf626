"""Pins of the CPU oracle against what the pages and the mathematics fix.

No GPU.  Each check is chosen so that a plausible slip in the oracle (a
dropped term, a wrong sign or index, a transposed operand, C read when
beta == 0, a wrong storage-order formula) fails at least one of them; the
last test plants such slips in a copy of the oracle and checks that they are
caught.
"""
import itertools
import os
import subprocess
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import COL, ROW
from oracle.tiled_counted import naive_counted, tiled_counted, tiled_traffic_bytes
from golden.fixtures import read as read_fixture

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


# --------------------------------------------------------------------------
# helpers (storage layout only -- no GEMM arithmetic)
# --------------------------------------------------------------------------
def store(X, order, pad=0, dtype=np.float32):
    """Lay the logical R x Q matrix X out in ``order`` with ld = minimal + pad.

    Returns (flat buffer, ld)."""
    X = np.asarray(X)
    R, Q = X.shape
    if order == ROW:
        ld = Q + pad
        buf = np.zeros((max(R, 1), ld), dtype=dtype)
        buf[:R, :Q] = X
    else:
        ld = R + pad
        buf = np.zeros((max(Q, 1), ld), dtype=dtype)
        buf[:Q, :R] = X.T
    return np.ascontiguousarray(buf.reshape(-1)), max(ld, 1)


def bf16_bits(X):
    """float32 values -> bf16 bit patterns (round to nearest even, torch CPU)."""
    t = torch.from_numpy(np.ascontiguousarray(X, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f32(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def run_oracle(A, B, alpha=1.0, beta=0.0, C=None, orders=(ROW, ROW, ROW), bf16=False, pad=0,
               nthreads=0):
    """bf16: False (FP32 inputs), True or "bf16" (BF16 inputs), "f16" (FP16 inputs)."""
    A = np.asarray(A, dtype=np.float32)
    B = np.asarray(B, dtype=np.float32)
    M, K = A.shape
    N = B.shape[1]
    oa, ob, oc = orders
    if bf16 == "f16":
        abuf, lda = store(A.astype(np.float16), oa, pad, np.float16)
        bbuf, ldb = store(B.astype(np.float16), ob, pad, np.float16)
    elif bf16:
        abuf, lda = store(bf16_bits(A).reshape(A.shape), oa, pad, np.uint16)
        bbuf, ldb = store(bf16_bits(B).reshape(B.shape), ob, pad, np.uint16)
    else:
        abuf, lda = store(A, oa, pad)
        bbuf, ldb = store(B, ob, pad)
    if C is not None:
        cbuf, ldc = store(np.asarray(C, dtype=np.float32), oc, pad)
    else:
        cbuf, ldc = None, 1
    return oracle.gemm(M, N, K, alpha, abuf, lda, oa, bbuf, ldb, ob, beta, cbuf, ldc, oc,
                       nthreads=nthreads)


def exact_reference(A, B, alpha, beta, C):
    """Independent exact loop over Python integers / fractions."""
    M, K = len(A), len(A[0]) if len(A) else 0
    N = len(B[0]) if len(B) else 0
    out = [[None] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            s = sum(Fraction(int(A[i][k])) * Fraction(int(B[k][j])) for k in range(K))
            v = Fraction(alpha) * s
            if beta != 0:
                v += Fraction(beta) * Fraction(int(C[i][j]))
            out[i][j] = v
    return out


def small_ints(rng, shape, lo=-4, hi=4):
    return rng.integers(lo, hi + 1, size=shape).astype(np.float32)


# --------------------------------------------------------------------------
# 1. The hand-traced 4x4 product with 2x2 tiles
# --------------------------------------------------------------------------
def _eval_expr(expr, A, B):
    """Evaluate 'A00*B00 + A01*B10' with the given integer matrices."""
    total = 0
    for term in expr.split("+"):
        fa, fb = [f.strip() for f in term.split("*")]
        assert fa[0] == "A" and fb[0] == "B"
        total += int(A[int(fa[1])][int(fa[2])]) * int(B[int(fb[1])][int(fb[2])])
    return total


def test_hand_trace_4x4_partial_sums():
    g = read_fixture("p5_4x4_2x2_tiles.txt")
    # distinct small integers so that a swapped index changes the value
    A = [[1, 2, 3, 4], [5, 6, 7, 8], [-1, -2, -3, -4], [2, 0, -1, 3]]
    B = [[3, -1, 2, 0], [1, 4, -2, 5], [0, 2, 1, -3], [-2, 1, 0, 2]]
    # worked by hand from the first K step of the top-left tile:
    # acc00 = 1*3 + 2*1 = 5, acc01 = 1*-1 + 2*4 = 7,
    # acc10 = 5*3 + 6*1 = 21, acc11 = 5*-1 + 6*4 = 19
    hand = {"acc00": 5, "acc01": 7, "acc10": 21, "acc11": 19}
    for key, value in hand.items():
        assert _eval_expr(g[key], A, B) == value
    trace = []
    C, _ = tiled_counted(A, B, 2, trace=trace)
    first = trace[0]
    assert (first.tile_row, first.tile_col, first.k0) == (0, 0, 0)
    assert first.acc == [[5, 7], [21, 19]]
    # C00 after the second step: 5 + 3*0 + 4*-2 = -3
    assert _eval_expr(g["C00"], A, B) == -3
    assert C[0][0] == -3
    D, _ = run_oracle(A, B)
    assert D[0, 0] == -3.0
    assert np.array_equal(D, np.array(C, dtype=np.float64))


def test_hand_trace_4x4_counts():
    g = {k: v for k, v in read_fixture("p5_4x4_2x2_tiles.txt").items() if not k.startswith(("acc", "C"))}
    rng = np.random.default_rng(1)
    A = small_ints(rng, (4, 4)).astype(int).tolist()
    B = small_ints(rng, (4, 4)).astype(int).tolist()
    trace = []
    _, tiled = tiled_counted(A, B, 2, trace=trace)
    _, naive = naive_counted(A, B)
    step = trace[0]
    assert step.reads == int(g["step_reads"])
    assert step.flops == int(g["step_flops"])
    assert 4 * step.reads == int(g["step_bytes"])
    steps_per_tile = 2
    tiles = 4
    assert tiled.reads == tiles * int(g["tile_reads"])
    assert tiled.writes == tiles * int(g["tile_writes"])
    assert tiled.flops == tiles * int(g["tile_flops"])
    assert sum(s.reads for s in trace[:steps_per_tile]) == int(g["tile_reads"])
    assert tiled.hbm_bytes // tiles == int(g["tile_bytes"])
    assert tiled.reads == int(g["total_reads"])
    assert tiled.writes == int(g["total_writes"])
    assert tiled.flops == int(g["total_flops"])
    assert tiled.hbm_bytes == int(g["total_bytes"])
    assert naive.reads == int(g["naive_reads"])
    assert naive.writes == int(g["naive_writes"])
    assert naive.flops == int(g["naive_flops"])
    assert naive.hbm_bytes == int(g["naive_bytes"])
    assert tiled.intensity == pytest.approx(float(g["intensity_tiled"]), abs=5e-7)
    assert naive.intensity == pytest.approx(float(g["intensity_naive"]), abs=5e-7)
    assert naive.hbm_bytes / tiled.hbm_bytes == pytest.approx(float(g["traffic_ratio"]))


# --------------------------------------------------------------------------
# 2. Tiled == naive == oracle, and the traffic formulas
# --------------------------------------------------------------------------
@pytest.mark.parametrize("n", [2, 4, 8])
def test_tiled_equals_naive_equals_oracle(n):
    rng = np.random.default_rng(100 + n)
    A = small_ints(rng, (n, n))
    B = small_ints(rng, (n, n))
    c_naive, cnt_naive = naive_counted(A.astype(int).tolist(), B.astype(int).tolist())
    D, _ = run_oracle(A, B)
    assert np.array_equal(D, np.array(c_naive, dtype=np.float64))
    for T in [t for t in range(1, n + 1) if n % t == 0]:
        c_tiled, cnt = tiled_counted(A.astype(int).tolist(), B.astype(int).tolist(), T)
        assert c_tiled == c_naive
        # counted traffic equals the closed form 8 n^3 / T + 4 n^2
        assert cnt.hbm_bytes == tiled_traffic_bytes(n, T)
        assert cnt.flops == 2 * n ** 3 == cnt_naive.flops
    assert cnt_naive.hbm_bytes == tiled_traffic_bytes(n, 1)


def test_traffic_tables_4096():
    g = read_fixture("p5_4096_fp32_traffic.txt")
    n = int(g["n"])
    flops = 2 * n ** 3
    assert flops == int(g["flops"])
    for T, key in [(1, "no_reuse"), (32, "T32"), (64, "T64"), (128, "T128")]:
        q = tiled_traffic_bytes(n, T)
        assert q == int(g["Q_" + key])
        assert round(flops / q, 6) == pytest.approx(float(g["I_" + key]), abs=1e-9)
    one_pass = 4 * (n * n + n * n) + 4 * n * n  # A and B read once, C written once
    assert one_pass == int(g["Q_one_pass"])
    assert round(flops / one_pass, 3) == pytest.approx(float(g["I_one_pass"]), abs=1e-9)
    # exercise 3: a 64 x 64 output tile over K = 4096 reads 4*K*(64+64) bytes
    # whatever the K slice width, and writes its tile once
    for bk in (32, 64):
        steps = n // bk
        assert steps * 4 * bk * (64 + 64) == int(g["ex3_tile_input_bytes"])
    assert 4 * 64 * 64 == int(g["ex3_tile_write_bytes"])


# --------------------------------------------------------------------------
# 3. Closed forms: identity, permutation, alpha/beta, K = 0
# --------------------------------------------------------------------------
@pytest.mark.parametrize("bf16", [False, True, "f16"])
@pytest.mark.parametrize("orders", [(ROW, ROW, ROW), (COL, ROW, COL), (ROW, COL, ROW), (COL, COL, COL)])
def test_identity_and_permutation(bf16, orders):
    rng = np.random.default_rng(7)
    M, K = 13, 9
    X = rng.uniform(-1, 1, size=(M, K)).astype(np.float32)
    if bf16 == "f16":
        X = X.astype(np.float16).astype(np.float32)
    elif bf16:
        X = bits_to_f32(bf16_bits(X)).reshape(M, K)
    D, _ = run_oracle(X, np.eye(K, dtype=np.float32), orders=orders, bf16=bf16)
    assert np.array_equal(D.astype(np.float32), X)
    D, _ = run_oracle(np.eye(M, dtype=np.float32), X, orders=orders, bf16=bf16)
    assert np.array_equal(D.astype(np.float32), X)
    perm = rng.permutation(M)
    P = np.zeros((M, M), dtype=np.float32)
    P[np.arange(M), perm] = 1.0  # (P X)_i = X_perm[i]
    D, _ = run_oracle(P, X, orders=orders, bf16=bf16)
    assert np.array_equal(D.astype(np.float32), X[perm])
    # X P^T permutes columns
    Q = np.zeros((K, K), dtype=np.float32)
    cperm = rng.permutation(K)
    Q[cperm, np.arange(K)] = 1.0  # (X Q)_{:, j} = X_{:, cperm[j]}
    D, _ = run_oracle(X, Q, orders=orders, bf16=bf16)
    assert np.array_equal(D.astype(np.float32), X[:, cperm])


def test_alpha_beta_closed_forms():
    rng = np.random.default_rng(11)
    M, N, K = 7, 5, 6
    A = rng.uniform(-1, 1, size=(M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(K, N)).astype(np.float32)
    C = rng.uniform(-1, 1, size=(M, N)).astype(np.float32)
    # A = 0  =>  D = beta * C exactly
    D, S = run_oracle(np.zeros_like(A), B, alpha=1.5, beta=-0.25, C=C)
    assert np.array_equal(D, -0.25 * C.astype(np.float64))
    assert np.all(S == 0)
    # beta = 0: C is never read, even if it holds NaN
    Cnan = np.full((M, N), np.nan, dtype=np.float32)
    D0, _ = run_oracle(A, B)
    D, _ = run_oracle(A, B, beta=0.0, C=Cnan)
    assert not np.isnan(D).any() and np.array_equal(D, D0)
    # alpha = 2^p scales the result exactly
    for p in (-3, 1, 5):
        D, S = run_oracle(A, B, alpha=2.0 ** p)
        assert np.array_equal(D, (2.0 ** p) * D0)
    # alpha = 0: A and B are not read; D = beta * C
    Anan = np.full((M, K), np.nan, dtype=np.float32)
    D, _ = run_oracle(Anan, B, alpha=0.0, beta=2.0, C=C)
    assert np.array_equal(D, 2.0 * C.astype(np.float64))
    # K = 0: empty sum
    D, S = run_oracle(np.zeros((M, 0), np.float32), np.zeros((0, N), np.float32), alpha=1.0,
                      beta=0.5, C=C)
    assert np.array_equal(D, 0.5 * C.astype(np.float64)) and np.all(S == 0)
    # linearity in C: beta*C adds on top of the alpha*AB result
    D1, _ = run_oracle(A, B, alpha=0.5, beta=1.0, C=C)
    D2, _ = run_oracle(A, B, alpha=0.5)
    assert np.allclose(D1 - D2, C.astype(np.float64), rtol=0, atol=1e-15)


def test_transpose_identity():
    """(A B)^T = B^T A^T: the oracle computed both ways agrees exactly on integers."""
    rng = np.random.default_rng(12)
    A = small_ints(rng, (6, 4))
    B = small_ints(rng, (4, 9))
    D, _ = run_oracle(A, B)
    Dt, _ = run_oracle(B.T.copy(), A.T.copy())
    assert np.array_equal(D.T, Dt)


# --------------------------------------------------------------------------
# 4. Brute force over tiny shapes and all storage orders
# --------------------------------------------------------------------------
@pytest.mark.parametrize("bf16", [False, True, "f16"])
def test_brute_force_tiny(bf16):
    rng = np.random.default_rng(2024 + (2 if bf16 == "f16" else int(bf16)))
    shapes = list(itertools.product(range(1, 6), repeat=3))
    checked = 0
    for (M, N, K) in shapes:
        A = small_ints(rng, (M, K))
        B = small_ints(rng, (K, N))
        C = small_ints(rng, (M, N))
        for orders in itertools.product((ROW, COL), repeat=3):
            for alpha, beta in ((1.0, 0.0), (1.5, -0.25)):
                pad = (M + N + K) % 3
                D, S = run_oracle(A, B, alpha, beta, C if beta else None, orders, bf16, pad)
                want = exact_reference(A, B, alpha, beta, C)
                got = [[Fraction(float(D[i, j])) for j in range(N)] for i in range(M)]
                assert got == want, (M, N, K, orders, alpha, beta)
                s_want = np.abs(alpha * (A[:, :, None] * B[None, :, :])).sum(axis=1)
                assert np.array_equal(S, s_want.astype(np.float64))
                checked += 1
    assert checked == len(shapes) * 8 * 2


def test_f16_widening_matches_every_bit_pattern():
    """Column of all 65536 binary16 patterns times 1: D holds each value exactly."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = bits.view(np.float16)
    finite = ~np.isnan(vals)
    A = np.ascontiguousarray(vals[finite]).reshape(-1, 1)
    one = np.ones((1, 1), dtype=np.float16)
    M = A.shape[0]
    D, _ = oracle.gemm(M, 1, 1, 1.0, A.reshape(-1), 1, ROW, one.reshape(-1), 1, ROW)
    want = A.reshape(-1).astype(np.float64)  # numpy's binary16 -> double conversion
    assert np.array_equal(D.reshape(-1), want)
    # NaN patterns give NaN
    nan_bits = np.ascontiguousarray(vals[~finite][:64])
    D, _ = oracle.gemm(nan_bits.shape[0], 1, 1, 1.0, nan_bits, 1, ROW, one.reshape(-1), 1, ROW)
    assert np.isnan(D).all()


def test_rounding_against_exact_sum():
    """Random FP32 data: the double result is within the double rounding bound of the exact sum."""
    rng = np.random.default_rng(5)
    M, N, K = 3, 4, 37
    A = rng.uniform(-1, 1, size=(M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(K, N)).astype(np.float32)
    C = rng.uniform(-1, 1, size=(M, N)).astype(np.float32)
    alpha, beta = 1.5, -0.25
    D, S = run_oracle(A, B, alpha, beta, C)
    u = Fraction(1, 2 ** 53)
    for i in range(M):
        for j in range(N):
            exact = Fraction(alpha) * sum(Fraction(float(A[i, k])) * Fraction(float(B[k, j]))
                                          for k in range(K)) + Fraction(beta) * Fraction(float(C[i, j]))
            bound = (K + 2) * u * (Fraction(S[i, j]) + abs(Fraction(beta) * Fraction(float(C[i, j]))))
            assert abs(Fraction(float(D[i, j])) - exact) <= bound


def test_points_and_threads_agree():
    rng = np.random.default_rng(9)
    M, N, K = 33, 29, 40
    A = rng.uniform(-1, 1, size=(M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(K, N)).astype(np.float32)
    C = rng.uniform(-1, 1, size=(M, N)).astype(np.float32)
    D1, S1 = run_oracle(A, B, 1.5, -0.25, C, orders=(COL, ROW, COL), nthreads=1)
    D8, S8 = run_oracle(A, B, 1.5, -0.25, C, orders=(COL, ROW, COL), nthreads=8)
    assert np.array_equal(D1, D8) and np.array_equal(S1, S8)
    abuf, lda = store(A, COL)
    bbuf, ldb = store(B, ROW)
    cbuf, ldc = store(C, COL)
    I = rng.integers(0, M, 200)
    J = rng.integers(0, N, 200)
    Dp, Sp = oracle.gemm_points(M, N, K, 1.5, abuf, lda, COL, bbuf, ldb, ROW, -0.25, cbuf, ldc,
                                COL, I, J, nthreads=3)
    assert np.array_equal(Dp, D1[I, J]) and np.array_equal(Sp, S1[I, J])


def test_rejects_bad_arguments():
    A = np.zeros(4, np.float32)
    with pytest.raises(ValueError):
        oracle.gemm(-1, 2, 2, 1.0, A, 2, ROW, A, 2, ROW)
    with pytest.raises(ValueError):  # beta != 0 needs C
        oracle.gemm(2, 2, 2, 1.0, A, 2, ROW, A, 2, ROW, beta=1.0, C=None)
    with pytest.raises(ValueError):  # point out of range
        oracle.gemm_points(2, 2, 2, 1.0, A, 2, ROW, A, 2, ROW, 0.0, None, 1, ROW, [2], [0])


# --------------------------------------------------------------------------
# 5. Planted mistakes are caught (mutants of the oracle, built on the CPU)
# --------------------------------------------------------------------------
MUTANTS = {
    "dropped first term": ("for (int64_t k = 0; k < p->K; ++k)", "for (int64_t k = 1; k < p->K; ++k)"),
    "wrong sign of beta*C": ("d = d + p->beta * c;", "d = d - p->beta * c;"),
    "transposed A": ("offset(p->order_a, p->lda, i, k)", "offset(p->order_a, p->lda, k, i)"),
    "column-major formula swapped": ("r * ld + q : r + q * ld", "r + q * ld : r * ld + q"),
    "C read with the wrong order": ("offset(p->order_c, p->ldc, i, j)", "offset(ORACLE_ROW, p->ldc, i, j)"),
    "FP16 exponent bias off by one": ("exponent - 25", "exponent - 24"),
    "FP16 implicit bit dropped": ("(double)(1024 + fraction)", "(double)(fraction)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(name, tmp_path):
    import ctypes
    src = open(os.path.join(ROOT, "oracle", "gemm_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1
    mutated = src.replace(old, new)
    cfile = tmp_path / "mutant.c"
    cfile.write_text(mutated)
    lib_path = tmp_path / "libmutant.so"
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", str(lib_path), str(cfile), "-lm"], check=True)
    lib = ctypes.CDLL(str(lib_path))
    i64, dbl, vp, ip = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
    lib.oracle_gemm.argtypes = [ip, i64, i64, i64, dbl, vp, i64, ip, vp, i64, ip, dbl, vp, i64,
                                ip, vp, vp, ip]
    lib.oracle_gemm.restype = ip
    rng = np.random.default_rng(3)
    caught = False
    for (M, N, K) in [(3, 4, 5), (4, 4, 4), (5, 2, 3)]:
        A = small_ints(rng, (M, K))
        B = small_ints(rng, (K, N))
        C = small_ints(rng, (M, N))
        for orders in itertools.product((ROW, COL), repeat=3):
            for in_type, dt in ((0, np.float32), (2, np.float16)):  # FP32 and FP16 inputs
                abuf, lda = store(A.astype(dt), orders[0], dtype=dt)
                bbuf, ldb = store(B.astype(dt), orders[1], dtype=dt)
                cbuf, ldc = store(C, orders[2])
                D = np.zeros((M, N))
                S = np.zeros((M, N))
                lib.oracle_gemm(in_type, M, N, K, 1.5, abuf.ctypes.data, lda, orders[0],
                                bbuf.ctypes.data, ldb, orders[1], -0.25, cbuf.ctypes.data, ldc,
                                orders[2], D.ctypes.data, S.ctypes.data, 1)
                if not np.isfinite(D).all():  # a mutant reading the wrong elements
                    caught = True
                    continue
                want = exact_reference(A, B, 1.5, -0.25, C)
                got = [[Fraction(float(D[i, j])) for j in range(N)] for i in range(M)]
                if got != want:
                    caught = True
    assert caught, f"mutant '{name}' survived the brute-force pin"
