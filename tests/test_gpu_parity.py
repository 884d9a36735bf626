"""GPU parity: the CUDA library against the CPU oracle, element by element.

Every test calls the C ABI (through the package binding) on seeded inputs
and compares with the oracle on the same bits:
  * FP32:  |D - D_ref| <= 1e-5 * sum_k|alpha A_ik B_kj| + 1e-6 * |beta C_ij|
  * BF16:  |D - D_ref| <= 4e-3 * sum_k|alpha A_ik B_kj| + 1e-6
  * small-integer inputs (every partial sum exact in FP32): bit-exact.
Full-size workloads are checked on sampled entries (whole rows and columns,
tile-boundary entries, corners, random entries) that the oracle computes one
by one; moderate sizes spanning several tiles with ragged tails are checked
in full, together with a guard band around D.
"""
import itertools

import numpy as np
import pytest
import torch

import dense_gemm_08_gb300 as lib
from dense_gemm_08_gb300.inputs import COL, ROW, WORKLOADS, Workload, make_inputs
from gemm_harness import (assert_within, c_logical, check_canary, logical_d, oracle_full,
                          oracle_points, run_gpu, sample_points)

pytestmark = pytest.mark.gpu

ORDERS = list(itertools.product((ROW, COL), repeat=3))


def full_check(w, inp, pad_d=0, expect_kernel=None):
    Dbuf, ldd, name = run_gpu(w, inp, pad_d=pad_d)
    if expect_kernel is not None:
        assert name.startswith(expect_kernel), name
    D = logical_d(w, Dbuf)
    ref, S = oracle_full(w, inp)
    ratio = assert_within(w, D, ref, S, c_logical(w, inp))
    if pad_d:
        check_canary(w, Dbuf)
    return D, ref, ratio


def sampled_check(w, inp, rows, cols, n_random=4000, seed=0):
    Dbuf, ldd, name = run_gpu(w, inp)
    D = logical_d(w, Dbuf)
    rng = np.random.default_rng(seed)
    I, J = sample_points(w.M, w.N, rng, n_random, rows, cols)
    ref, S = oracle_points(w, inp, I, J)
    C = c_logical(w, inp)
    Cv = C[I, J] if C is not None else None
    assert np.isfinite(D).all(), f"{w.name}: non-finite output"
    return assert_within(w, D[I, J], ref, S, Cv, "sampled"), name


# ---------------------------------------------------------------- the configs
def test_f32_256_full():
    w = WORKLOADS["f32_256"]
    full_check(w, make_inputs(w), pad_d=3, expect_kernel="sgemm_cluster<f32")


def test_f32_256_small_integers_bit_exact():
    w = WORKLOADS["f32_256_int"]
    inp = make_inputs(w)
    Dbuf, _, _ = run_gpu(w, inp)
    ref, _ = oracle_full(w, inp)
    assert np.array_equal(logical_d(w, Dbuf), ref.astype(np.float32))


@pytest.mark.parametrize("name", ["f32_4096", "bf16_8192", "bf16_mlp"])
def test_full_size_config_sampled(name):
    w = WORKLOADS[name]
    inp = make_inputs(w)
    ratio, kernel = sampled_check(w, inp, rows=(0, 1, w.M // 2 + 3, w.M - 1),
                                  cols=(0, w.N // 3 + 1, w.N - 1))
    if w.dtype == "bf16":
        assert kernel.startswith("gemm_bf16_tc<pair")


@pytest.mark.parametrize("name", sorted(k for k in WORKLOADS if k.startswith("odd_")))
def test_odd_shape_sweep(name):
    w = WORKLOADS[name]
    inp = make_inputs(w)
    if w.M * w.N * w.K <= 64 * 1024 * 1024:
        full_check(w, inp)
    else:
        sampled_check(w, inp, rows=(0, w.M // 2, w.M - 1), cols=(0, w.N - 1), n_random=3000)


# ------------------------------------------- moderate sizes, checked in full
MODERATE = (300, 600, 200)  # 3 x 3 tensor-core tiles with ragged M, N and K tails


@pytest.mark.parametrize("orders", ORDERS)
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_all_orders_full(dtype, orders):
    M, N, K = MODERATE
    w = Workload(f"mod_{dtype}", M, N, K, 1.5, -0.25, dtype, *orders)
    inp = make_inputs(w, seed=1, pad=3, ld_multiple=8)
    expect = {"f32": "sgemm_cluster<f32", "bf16": "gemm_bf16_tc", "f16": "gemm_f16_tc"}[dtype]
    full_check(w, inp, pad_d=5, expect_kernel=expect)


# Big enough for the CTA-pair variant (>= 100 tiles of 256 x 256), ragged in
# M, N and K, so both CTAs of a pair see partial tiles.  With 76 resident
# pairs its last round holds 34 tiles, each split into two N halves.
PAIR_SHAPE = (2500, 2600, 136)


@pytest.mark.parametrize("orders", ORDERS)
def test_cta_pair_variant_all_orders_full(orders):
    M, N, K = PAIR_SHAPE
    w = Workload("pair", M, N, K, 1.5, -0.25, "bf16", *orders)
    inp = make_inputs(w, seed=11, pad=5, ld_multiple=8)
    full_check(w, inp, pad_d=3, expect_kernel="gemm_bf16_tc<pair")
    assert "direct" not in lib.gemm_last_kernel()


# Fewer 128 x 256 tiles than SMs and a long K: the tensor-core kernel splits
# each tile's K range over several CTAs and the last one adds the pieces.
TC_SPLIT_SHAPE = (300, 600, 2048)


@pytest.mark.parametrize("orders", ORDERS)
def test_tc_split_k_all_orders_full(orders):
    M, N, K = TC_SPLIT_SHAPE
    w = Workload("tc_splitk", M, N, K, 1.5, -0.25, "bf16", *orders)
    inp = make_inputs(w, seed=18, pad=3, ld_multiple=8)
    full_check(w, inp, pad_d=3, expect_kernel="gemm_bf16_tc<splitk,")


def test_tc_split_k_deterministic_and_exact_on_integers():
    M, N, K = TC_SPLIT_SHAPE
    w = Workload("tc_splitk_int", M, N, K, 1.0, 0.0, "bf16", ROW, COL, ROW, dist="int")
    inp = make_inputs(w, seed=19)
    D1, _, name = run_gpu(w, inp)
    assert name.startswith("gemm_bf16_tc<splitk,"), name
    ref, _ = oracle_full(w, inp)
    assert np.array_equal(logical_d(w, D1), ref.astype(np.float32))
    w = w.with_(dist="normal", alpha=0.5, beta=1.0)
    inp = make_inputs(w, seed=20)
    D1, _, _ = run_gpu(w, inp)
    D2, _, _ = run_gpu(w, inp)
    assert torch.equal(D1, D2)


# The split-K cluster size ks is the largest of SMs // tiles, K blocks // 4
# and 8 whose clusters (one per 128 x 256 tile) are all resident at once.
# On 152 SMs these shapes ask for every size from 2 to 8 (fewer where a GPC
# cannot hold that many clusters), with ragged M, N and K: warps whose rows
# are all past M (M = 33), a last tile holding one partial 32-column chunk
# (N = 520), a partial last K block, C and D through TMA boxes or row
# copies.  (M, N, K, pad_d, beta)
CLUSTER_SPLIT_SHAPES = [
    (100, 200, 2048, 0, -0.25),    # 1 tile, 32 K blocks: 8 pieces
    (33, 520, 4095, 3, 0.5),       # 3 tiles: 8 pieces, K blocks 64 (last partial)
    (2432, 200, 2048, 0, 1.0),     # 19 tiles: 8 (or fewer, where 19 clusters of 8 do not fit)
    (2688, 250, 1800, 3, -0.25),   # 21 tiles: 7
    (3200, 256, 1536, 0, 0.0),     # 25 tiles: 6 (24 K blocks)
    (3840, 230, 2000, 0, -0.25),   # 30 tiles: 5
    (640, 1280, 999, 3, 1.0),      # 25 tiles, 16 K blocks: 4
    (1200, 1200, 2000, 0, -0.25),  # 50 tiles: 3
    (1000, 1000, 640, 3, 0.0),     # 32 tiles, 10 K blocks: 2
    (300, 600, 200, 0, -0.25),     # 4 K blocks: no split
]


@pytest.mark.parametrize("shape", CLUSTER_SPLIT_SHAPES, ids=[f"{m}x{n}x{k}" for m, n, k, _, _ in
                                                            CLUSTER_SPLIT_SHAPES])
def test_tc_cluster_split_sizes_full(shape):
    M, N, K, pad_d, beta = shape
    w = Workload("tc_cluster", M, N, K, 1.5, beta, "bf16", ROW, COL, ROW)
    inp = make_inputs(w, seed=M + N + K, ld_multiple=8)
    D, ref, _ = full_check(w, inp, pad_d=pad_d, expect_kernel="gemm_bf16_tc")
    name = lib.gemm_last_kernel()
    tiles = -(-M // 128) * -(-N // 256)
    want_max = min(torch.cuda.get_device_properties(0).multi_processor_count // tiles,
                   -(-K // 64) // 4, 8)
    if want_max < 2:
        assert name == "gemm_bf16_tc", name
    else:
        assert name.startswith("gemm_bf16_tc<splitk,x"), name
        ks = int(name[len("gemm_bf16_tc<splitk,x"):-1])
        assert 2 <= ks <= want_max, name
        # the pieces are added in K order: a second call gives the same bits
        D2, _, _ = run_gpu(w, inp, pad_d=pad_d)
        assert np.array_equal(logical_d(w, D2), D)


# N <= 128 (after the column-major normalisation): single CTAs take a 64- or
# 128-row B box and N = 64 / 128 MMAs, with the ring cut into 8 or 6
# stages; with few tiles the K range is split over a cluster as well.
# Both B orders (K-contiguous: one narrow box; N-contiguous: one or two
# 64-column boxes), N at and around the box widths, ragged M and K.
NARROW_N_SHAPES = [
    (1000, 64, 777), (1000, 65, 300), (1000, 128, 520), (2000, 33, 1000), (700, 1, 256),
    # N <= 32 with a K-contiguous B: 16 or 32 rows of B per stage, the
    # other rows stale (they reach only columns past N)
    (1500, 7, 600), (1500, 16, 600), (1500, 17, 600), (1500, 32, 600),
    (300, 100, 2048),  # 3 tiles: split-K over a cluster with the narrow box
    (200, 9, 3000),  # 2 tiles: split-K with a 16-row B box
]


@pytest.mark.parametrize("b_order", [COL, ROW])
@pytest.mark.parametrize("shape", NARROW_N_SHAPES, ids=[f"{m}x{n}x{k}" for m, n, k in NARROW_N_SHAPES])
def test_tc_narrow_n_tiles_full(shape, b_order):
    M, N, K = shape
    w = Workload("tc_narrow", M, N, K, 1.5, -0.25, "bf16", ROW, b_order, ROW)
    inp = make_inputs(w, seed=M + 3 * N + K, ld_multiple=8)
    full_check(w, inp, pad_d=3, expect_kernel="gemm_bf16_tc")
    # deterministic: a second call gives the same bits
    D1, _, _ = run_gpu(w, inp)
    D2, _, _ = run_gpu(w, inp)
    assert torch.equal(D1, D2)


# M <= 64: single CTAs load 16, 32 or 64 rows of a K-contiguous A (one
# 64-row box of an M-contiguous A); the tile's other rows hold stale shared
# memory and must not reach D.  M at and around each box height, both A
# orders, with and without the cluster split-K, beta != 0 (C read).
SMALL_M = [1, 7, 16, 17, 32, 33, 64]


@pytest.mark.parametrize("a_order", [ROW, COL])
@pytest.mark.parametrize("M", SMALL_M)
def test_tc_small_m_a_box_full(M, a_order):
    for N, K in [(600, 1000), (2000, 96)]:  # split over a cluster; K = 96: no split
        w = Workload("tc_small_m", M, N, K, 1.5, -0.25, "bf16", a_order, COL, ROW)
        inp = make_inputs(w, seed=M * 7 + N + K, ld_multiple=8)
        full_check(w, inp, pad_d=3, expect_kernel="gemm_bf16_tc")


@pytest.mark.parametrize("orders", [(ROW, COL, ROW), (COL, ROW, COL)])
def test_f16_pair_and_split_variants_full(orders):
    for shape, kernel in [(PAIR_SHAPE, "gemm_f16_tc<pair"), (TC_SPLIT_SHAPE, "gemm_f16_tc<splitk,")]:
        M, N, K = shape
        w = Workload("f16var", M, N, K, 1.5, -0.25, "f16", *orders)
        inp = make_inputs(w, seed=22, pad=5, ld_multiple=8)
        full_check(w, inp, pad_d=3, expect_kernel=kernel)


def test_f16_unaligned_operands_use_cuda_core_path():
    w = Workload("f16unal", 150, 270, 101, 1.5, -0.25, "f16", ROW, COL, ROW)
    inp = make_inputs(w, seed=23)  # lda = ldb = 101
    full_check(w, inp, pad_d=1, expect_kernel="sgemm_simt<f16")


def test_f16_8192_sampled():
    w = WORKLOADS["f16_8192"]
    inp = make_inputs(w)
    ratio, kernel = sampled_check(w, inp, rows=(0, w.M // 2 + 3, w.M - 1), cols=(0, w.N - 1))
    assert kernel.startswith("gemm_f16_tc<pair")


def test_cta_pair_variant_small_integers_bit_exact():
    w = Workload("pair_int", 2304, 2560, 1000, 1.0, 0.0, "bf16", ROW, COL, ROW, dist="int")
    inp = make_inputs(w, seed=12)
    Dbuf, _, name = run_gpu(w, inp)
    assert name.startswith("gemm_bf16_tc<pair,direct")  # beta = 0, 32-byte rows
    ref, _ = oracle_full(w, inp)
    assert np.array_equal(logical_d(w, Dbuf), ref.astype(np.float32))
    # the staged epilogue on the same problem (ldd not a multiple of 8)
    Dbuf, _, name = run_gpu(w, inp, pad_d=3)
    assert name.startswith("gemm_bf16_tc<pair") and "direct" not in name, name
    assert np.array_equal(logical_d(w, Dbuf), ref.astype(np.float32))


# The CTA-pair kernel's last round: with 76 resident pairs these shapes leave
# 28, 20 and 14 tiles for it.  28 and 20 fill more than a quarter of the
# pairs: each tile is split into its two N halves (whole K, no partial
# sums); 14 is split into 4 K ranges whose partial sums the last piece to
# finish adds.  Ragged M, N and K in the first.
TAIL_SHAPES = [(2000, 3300, 777), (2048, 3072, 768), (2304, 2560, 1024)]
TAIL_KIND = {TAIL_SHAPES[0]: "split-n-tail", TAIL_SHAPES[1]: "split-n-tail",
             TAIL_SHAPES[2]: "split-tail"}


def _pairs_resident():
    return torch.cuda.get_device_properties(0).multi_processor_count // 2


@pytest.mark.parametrize("orders", ORDERS)
def test_cta_pair_split_tail_all_orders_full(orders):
    M, N, K = TAIL_SHAPES[0]
    w = Workload("pair_tail", M, N, K, 1.5, -0.25, "bf16", *orders)
    inp = make_inputs(w, seed=26, pad=3, ld_multiple=8)
    D, _, _ = full_check(w, inp, pad_d=3, expect_kernel="gemm_bf16_tc<pair")
    if _pairs_resident() == 76:
        assert lib.gemm_last_kernel() == "gemm_bf16_tc<pair,split-n-tail>"


@pytest.mark.parametrize("orders", ORDERS)
def test_cta_pair_split_k_tail_all_orders_full(orders):
    M, N, K = TAIL_SHAPES[2]
    w = Workload("pair_tail_k", M, N - 3, K - 5, 1.5, -0.25, "bf16", *orders)
    inp = make_inputs(w, seed=28, pad=3, ld_multiple=8)
    # ldd = 2561 (row-major D) or 2308 (column-major): rows not on 32 bytes,
    # so the staged epilogue runs
    full_check(w, inp, pad_d=4, expect_kernel="gemm_bf16_tc<pair")
    if _pairs_resident() == 76:
        assert lib.gemm_last_kernel() == "gemm_bf16_tc<pair,split-tail>"


@pytest.mark.parametrize("shape", TAIL_SHAPES[1:])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_cta_pair_split_tail_pieces_full(shape, dtype):
    M, N, K = shape
    w = Workload("pair_tail", M, N, K, 0.5, 1.0, dtype, ROW, COL, ROW)
    inp = make_inputs(w, seed=27, ld_multiple=8)
    full_check(w, inp, pad_d=4, expect_kernel=f"gemm_{dtype}_tc<pair")


def test_cta_pair_split_tail_deterministic():
    M, N, K = TAIL_SHAPES[2]
    w = Workload("pair_tail_det", M, N, K, 0.5, 1.0, "bf16", ROW, COL, ROW)
    inp = make_inputs(w, seed=28)
    D1, _, name = run_gpu(w, inp)
    D2, _, _ = run_gpu(w, inp)
    assert name.startswith("gemm_bf16_tc<pair")
    assert torch.equal(D1, D2)


# Split-K on the CUDA-core path: few tiles (every tile split along K) and a
# last partial wave (only its tiles split); results must not depend on the
# order in which the pieces finish.
@pytest.mark.parametrize("orders", ORDERS)
def test_split_k_all_tiles_full(orders):
    w = Workload("splitk", 384, 384, 1000, 1.5, -0.25, "f32", *orders)
    inp = make_inputs(w, seed=13, pad=2)
    full_check(w, inp, pad_d=2, expect_kernel="sgemm_simt<f32")


def test_split_k_last_wave_full():
    w = Workload("splitk_tail", 2560, 2048, 512, 1.5, -0.25, "f32", ROW, ROW, ROW)
    inp = make_inputs(w, seed=14)
    full_check(w, inp, pad_d=1, expect_kernel="sgemm_simt<f32")


def test_split_k_bf16_fallback_full():
    # odd leading dimensions keep BF16 on the CUDA-core kernel, which splits K too
    w = Workload("splitk_bf16", 300, 200, 999, 1.5, -0.25, "bf16", ROW, COL, ROW)
    inp = make_inputs(w, seed=15, pad=2)  # lda = ldb = 1001: not a multiple of 8
    full_check(w, inp, expect_kernel="sgemm_simt<bf16")


@pytest.mark.parametrize("shape", [(384, 384, 1000), (2560, 2048, 512)])
def test_split_k_is_deterministic_and_exact_on_integers(shape):
    M, N, K = shape
    w = Workload("splitk_int", M, N, K, 1.0, 0.0, "f32", dist="int")
    inp = make_inputs(w, seed=16)
    D1, _, _ = run_gpu(w, inp)
    D2, _, _ = run_gpu(w, inp)
    assert torch.equal(D1, D2)
    ref, _ = oracle_full(w, inp)
    assert np.array_equal(logical_d(w, D1), ref.astype(np.float32))
    w = w.with_(dist="uniform")
    inp = make_inputs(w, seed=17)
    D1, _, _ = run_gpu(w, inp)
    D2, _, _ = run_gpu(w, inp)
    assert torch.equal(D1, D2)


@pytest.mark.parametrize("shape", [(257, 515, 1000), (128, 256, 64), (1, 1, 1), (129, 1, 77),
                                   (1, 300, 513), (640, 512, 8)])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_small_integers_bit_exact(dtype, shape):
    M, N, K = shape
    for orders in [(ROW, COL, ROW), (COL, ROW, ROW), (ROW, ROW, COL)]:
        w = Workload("int", M, N, K, 1.0, 0.0, dtype, *orders, dist="int")
        inp = make_inputs(w, seed=2, ld_multiple=8)
        Dbuf, _, _ = run_gpu(w, inp)
        ref, _ = oracle_full(w, inp)
        assert np.array_equal(logical_d(w, Dbuf), ref.astype(np.float32)), orders


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_tiny_shapes_brute_force(dtype):
    """Every (M, N, K) in {1..5, 9, 12} x {1..5}^2, every storage order, two
    (alpha, beta): M <= 8 takes the small-M kernel, M = 9 and 12 the tiled
    kernels (and a column-major D with N <= 5 the small-M kernel again)."""
    for M, N, K in itertools.product([1, 2, 3, 4, 5, 9, 12], range(1, 6), range(1, 6)):
        for orders in ORDERS:
            for alpha, beta in ((1.0, 0.0), (1.5, -0.25)):
                w = Workload("tiny", M, N, K, alpha, beta, dtype, *orders, dist="int")
                # ld a multiple of 8 keeps BF16 on the tensor-core path (M > 8)
                inp = make_inputs(w, seed=M * 100 + N * 10 + K, ld_multiple=8)
                Dbuf, _, name = run_gpu(w, inp)
                ref, _ = oracle_full(w, inp)
                got = logical_d(w, Dbuf)
                assert np.array_equal(got, ref.astype(np.float32)), (M, N, K, orders, alpha,
                                                                    beta, name)


# ------------------------------------------------------------- edge cases
def _dev(t):
    return t.to("cuda") if t is not None else None


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_empty_shapes_are_noops(dtype):
    fn = {"f32": lib.gemm_f32, "bf16": lib.gemm_bf16_f32acc, "f16": lib.gemm_f16_f32acc}[dtype]
    D = torch.full((4, 4), 7.0, device="cuda")
    assert fn(0, 4, 4, 1.0, None, 4, ROW, None, 4, ROW, 0.0, None, 4, D, 4, ROW) == 0
    assert fn(4, 0, 4, 1.0, None, 4, ROW, None, 4, ROW, 0.0, None, 4, D, 4, ROW) == 0
    assert lib.gemm_last_kernel() == ""
    torch.cuda.synchronize()
    assert torch.all(D == 7.0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_k_zero_and_alpha_zero_give_beta_c(dtype):
    w = Workload("kz", 70, 90, 0, 1.5, -0.25, dtype)
    inp = make_inputs(w, seed=3)
    full_check(w, inp, pad_d=2, expect_kernel="scale_c")
    # alpha = 0: A and B are not read (they hold NaN here)
    w = Workload("a0", 70, 90, 33, 0.0, 2.0, dtype)
    inp = make_inputs(w, seed=3)
    inp["A"] = torch.full_like(inp["A"], float("nan"))
    Dbuf, _, name = run_gpu(w, inp)
    assert name == "scale_c"
    assert np.array_equal(logical_d(w, Dbuf), (2.0 * inp["C_logical"]).numpy())


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_beta_zero_never_reads_c(dtype):
    w = Workload("b0", 200, 300, 64, 1.0, 0.0, dtype, ROW, COL, ROW)
    inp = make_inputs(w, seed=4, ld_multiple=8)
    A, B = _dev(inp["A"]), _dev(inp["B"])
    Cnan = torch.full((w.M, w.N), float("nan"), device="cuda")
    D = torch.empty((w.M, w.N), device="cuda")
    fn = {"f32": lib.gemm_f32, "bf16": lib.gemm_bf16_f32acc, "f16": lib.gemm_f16_f32acc}[dtype]
    fn(w.M, w.N, w.K, 1.0, A, inp["lda"], ROW, B, inp["ldb"], COL, 0.0, Cnan, w.N, D, w.N, ROW)
    torch.cuda.synchronize()
    assert torch.isfinite(D).all()


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_in_place_c_equals_d(dtype):
    w = Workload("inplace", 260, 520, 130, 0.5, 1.0, dtype, ROW, COL, ROW)
    inp = make_inputs(w, seed=5, ld_multiple=8)
    Dbuf, _, _ = run_gpu(w, inp, in_place=True)
    ref, S = oracle_full(w, inp)
    assert_within(w, logical_d(w, Dbuf), ref, S, c_logical(w, inp))


@pytest.mark.parametrize("shape", [PAIR_SHAPE, (2000, 3300, 777)])
def test_in_place_c_equals_d_pair_direct(shape):
    # the CTA pair's direct epilogue reads C and writes D through registers,
    # whole tiles and split tail tiles
    M, N, K = shape
    w = Workload("inplace_pair", M, N, K, 0.5, 1.0, "bf16", ROW, COL, ROW)
    inp = make_inputs(w, seed=7, ld_multiple=8)
    Dbuf, _, name = run_gpu(w, inp, in_place=True)
    assert name.startswith("gemm_bf16_tc<pair,direct"), name
    ref, S = oracle_full(w, inp)
    assert_within(w, logical_d(w, Dbuf), ref, S, c_logical(w, inp))


def test_bf16_unaligned_operands_use_cuda_core_path():
    """lda not a multiple of 8, and an operand starting 2 bytes off a 16-byte boundary."""
    w = Workload("unal", 150, 270, 101, 1.5, -0.25, "bf16", ROW, COL, ROW)
    inp = make_inputs(w, seed=6)  # lda = ldb = 101
    full_check(w, inp, pad_d=1, expect_kernel="sgemm_simt<bf16")
    # shift B by one element inside a bigger buffer
    inp2 = make_inputs(w, seed=6, ld_multiple=8)
    Bbig = torch.zeros(inp2["B"].numel() + 8, dtype=torch.bfloat16)
    Bbig[1:1 + inp2["B"].numel()] = inp2["B"].reshape(-1)
    A, Bd = _dev(inp2["A"]), Bbig.to("cuda")
    C = _dev(inp2["C"])
    D = torch.empty((w.M, w.N), device="cuda")
    lib.gemm_bf16_f32acc(w.M, w.N, w.K, w.alpha, A, inp2["lda"], ROW, Bd.data_ptr() + 2,
                         inp2["ldb"], COL, w.beta, C, inp2["ldc"], D, w.N, ROW)
    assert lib.gemm_last_kernel().startswith("sgemm_simt<bf16")
    torch.cuda.synchronize()
    ref, S = oracle_full(w, inp2)
    assert_within(w, D.cpu().numpy(), ref, S, c_logical(w, inp2))


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_tensor_core_ignores_operand_padding(dtype):
    """K (and M, N) not multiples of 8 with 16-byte-multiple leading dimensions:
    the tensor-core path must read only the matrix, never the padding (NaN here)."""
    for orders in ORDERS:
        w = Workload("padnan", 137, 261, 13, 1.5, -0.25, dtype, *orders)
        inp = make_inputs(w, seed=24, ld_multiple=8)
        for key in ("A", "B"):
            logical = inp[key + "_logical"]
            order = w.order_a if key == "A" else w.order_b
            store = inp[key]
            rows, cols = (logical.shape if order == ROW else logical.t().shape)
            mask = torch.ones_like(store, dtype=torch.bool)
            mask[:rows, :cols] = False
            store[mask] = float("nan")
        C = inp["C"]
        cmask = torch.ones_like(C, dtype=torch.bool)
        crow, ccol = (w.M, w.N) if w.order_cd == ROW else (w.N, w.M)
        cmask[:crow, :ccol] = False
        C[cmask] = float("nan")
        Dbuf, _, name = run_gpu(w, inp, pad_d=3)
        assert name.startswith("gemm_" + dtype + "_tc"), name
        D = logical_d(w, Dbuf)
        assert np.isfinite(D).all(), orders
        ref, S = oracle_full(w, inp)
        assert_within(w, D, ref, S, c_logical(w, inp), str(orders))
        check_canary(w, Dbuf)


@pytest.mark.parametrize("n", [601, 602, 603, 604, 608])
def test_tma_store_edges_stay_inside_d(n):
    """D with a 16-byte-multiple pitch but rows of N elements that are not
    whole 16-byte pieces: nothing may land past column N."""
    for dtype, beta in [("bf16", 0.0), ("bf16", -0.25), ("f16", 1.0)]:
        w = Workload("edge", 200, n, 96, 1.5, beta, dtype, ROW, COL, ROW)
        inp = make_inputs(w, seed=25, ld_multiple=8)
        pad = (-n) % 8 + 8  # ldd a multiple of 8 with spare columns
        full_check(w, inp, pad_d=pad)


# FP32 tile configurations: 128 x 256 (two waves, long K), 128 x 128 (few
# big tiles or short K), 256 x 64 (D at most 64 wide), 64 x 64 (small, K
# too long for the cluster kernel); ragged edges and stream-K tails in each.
SIMT_CFG_SHAPES = [(2560, 5120, 2048), (1100, 1300, 700), (700, 900, 500), (2000, 64, 777),
                   (3000, 33, 300), (130, 140, 1500)]


@pytest.mark.parametrize("shape", SIMT_CFG_SHAPES)
def test_f32_tile_configurations_full(shape):
    M, N, K = shape
    for orders in (ORDERS if M * N * K < 2e9 else ORDERS[:2]):
        w = Workload("f32cfg", M, N, K, 1.5, -0.25, "f32", *orders)
        inp = make_inputs(w, seed=M + N + K, pad=1)
        full_check(w, inp, pad_d=2, expect_kernel="sgemm_simt<f32")


def test_f32_unaligned_leading_dimensions():
    """Leading dimensions that are not multiples of 4 (scalar loads and stores)."""
    for orders in [(ROW, ROW, ROW), (COL, COL, COL)]:
        w = Workload("f32lds", 333, 257, 129, 1.5, -0.25, "f32", *orders)
        inp = make_inputs(w, seed=7, pad=1)
        full_check(w, inp, pad_d=1)


def test_invalid_arguments_are_rejected_before_launch():
    D = torch.zeros((8, 8), device="cuda")
    A = torch.zeros((8, 8), device="cuda")
    bad = [
        dict(M=-1),
        dict(lda=7),                    # row-major A needs lda >= K
        dict(ldd=7),                    # row-major D needs ldd >= N
        dict(order_a=2),
        dict(beta=1.0, C=None),         # beta != 0 needs C
        dict(A=None),
        dict(D=None),
        dict(A=A.data_ptr() + 2),       # misaligned FP32 pointer
    ]
    for change in bad:
        args = dict(M=8, N=8, K=8, alpha=1.0, A=A, lda=8, order_a=ROW, B=A, ldb=8, order_b=ROW,
                    beta=0.0, C=None, ldc=8, D=D, ldd=8, order_cd=ROW)
        args.update(change)
        st = lib.gemm_f32(args["M"], args["N"], args["K"], args["alpha"], args["A"],
                          args["lda"], args["order_a"], args["B"], args["ldb"], args["order_b"],
                          args["beta"], args["C"], args["ldc"], args["D"], args["ldd"],
                          args["order_cd"], check=False)
        assert st == lib.GEMM_ERR_INVALID_VALUE, change


def test_device_status_is_clean_after_runs():
    w = WORKLOADS["bf16_8192"].with_(M=1000, N=1000, K=1000)
    inp = make_inputs(w)
    run_gpu(w, inp)
    assert lib.gemm_last_device_status() == lib.GEMM_OK


def test_torch_helper_matches_oracle():
    w = Workload("helper", 300, 260, 90, 1.0, 0.0, "bf16", ROW, COL, ROW)
    inp = make_inputs(w, seed=8, ld_multiple=8)
    A = inp["A_logical"].to("cuda")
    Bt = inp["B_logical"].t().contiguous().to("cuda")  # N x K storage: B column-major
    D = lib.gemm(A, Bt.t())
    torch.cuda.synchronize()
    ref, S = oracle_full(w, inp)
    assert_within(w, D.cpu().numpy(), ref, S, None)


# ---------------------------------------------- the pair kernel's direct epilogue
# beta = 0 and D rows that start on 32 bytes (ldd a multiple of 8 FP32
# values): the CTA-pair kernel stores D from registers, with a 7-stage ring.
def _pad_to_32_bytes(w):
    cols = w.N if w.order_cd == ROW else w.M
    return 8 + (-cols) % 8  # ldd a multiple of 8, and a guard band


@pytest.mark.parametrize("orders", ORDERS)
def test_direct_epilogue_pair_all_orders_full(orders):
    M, N, K = PAIR_SHAPE
    w = Workload("pair_direct", M, N, K, 1.5, 0.0, "bf16", *orders)
    inp = make_inputs(w, seed=41, pad=5, ld_multiple=8)
    full_check(w, inp, pad_d=_pad_to_32_bytes(w), expect_kernel="gemm_bf16_tc<pair,direct")


@pytest.mark.parametrize("shape", TAIL_SHAPES)
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_direct_epilogue_split_tail_full(shape, dtype):
    M, N, K = shape
    w = Workload("tail_direct", M, N, K, 0.75, 0.0, dtype, ROW, COL, ROW)
    inp = make_inputs(w, seed=42, ld_multiple=8)
    full_check(w, inp, pad_d=_pad_to_32_bytes(w), expect_kernel=f"gemm_{dtype}_tc<pair,direct")
    if _pairs_resident() == 76:
        assert lib.gemm_last_kernel() == f"gemm_{dtype}_tc<pair,direct,{TAIL_KIND[shape]}>"


@pytest.mark.parametrize("shape", [TAIL_SHAPES[1], TAIL_SHAPES[2]])
def test_split_tails_small_integers_exact_and_deterministic(shape):
    # N-split tail (whole K per half) and K-split tail (partial sums added in
    # K order): bit-exact on small integers, run to run identical otherwise
    M, N, K = shape
    w = Workload("tail_int", M, N, K, 1.0, 0.0, "bf16", ROW, COL, ROW, dist="int")
    inp = make_inputs(w, seed=50)
    D1, _, name = run_gpu(w, inp)
    if _pairs_resident() == 76:
        assert name == f"gemm_bf16_tc<pair,direct,{TAIL_KIND[shape]}>", name
    ref, _ = oracle_full(w, inp)
    assert np.array_equal(logical_d(w, D1), ref.astype(np.float32))
    w = w.with_(dist="normal", alpha=0.5)
    inp = make_inputs(w, seed=51)
    D1, _, _ = run_gpu(w, inp)
    D2, _, _ = run_gpu(w, inp)
    assert torch.equal(D1, D2)


def test_direct_epilogue_split_tail_integers_exact_and_deterministic():
    w = Workload("tail_direct_int", 2048, 3072, 768, 1.0, 0.0, "bf16", ROW, COL, ROW, dist="int")
    inp = make_inputs(w, seed=43)
    D1, _, name = run_gpu(w, inp)
    assert name.startswith("gemm_bf16_tc<pair,direct")
    ref, _ = oracle_full(w, inp)
    assert np.array_equal(logical_d(w, D1), ref.astype(np.float32))
    w = w.with_(dist="normal", alpha=0.5)
    inp = make_inputs(w, seed=44)
    D1, _, _ = run_gpu(w, inp)
    D2, _, _ = run_gpu(w, inp)
    assert torch.equal(D1, D2)


@pytest.mark.parametrize("orders", ORDERS)
def test_direct_epilogue_with_c_all_orders_full(orders):
    # beta != 0 with C and D rows on 32 bytes: C is read into registers
    M, N, K = PAIR_SHAPE
    w = Workload("pair_direct_c", M, N, K, 1.5, -0.25, "bf16", *orders)
    inp = make_inputs(w, seed=45, pad=5, ld_multiple=8)
    full_check(w, inp, pad_d=_pad_to_32_bytes(w), expect_kernel="gemm_bf16_tc<pair,direct")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_direct_epilogue_with_c_split_tail_full(dtype):
    M, N, K = TAIL_SHAPES[0]  # ragged M, N and K
    w = Workload("tail_direct_c", M, N, K, 0.5, 1.0, dtype, COL, ROW, ROW)
    inp = make_inputs(w, seed=46, ld_multiple=8)
    full_check(w, inp, pad_d=_pad_to_32_bytes(w), expect_kernel=f"gemm_{dtype}_tc<pair,direct")
    if _pairs_resident() == 76:
        assert lib.gemm_last_kernel() == f"gemm_{dtype}_tc<pair,direct,split-n-tail>"


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_direct_epilogue_with_c_split_k_tail_full(dtype):
    M, N, K = TAIL_SHAPES[2]
    w = Workload("tail_direct_c_k", M, N, K - 7, 0.5, 1.0, dtype, ROW, ROW, ROW)
    inp = make_inputs(w, seed=52, ld_multiple=8)
    full_check(w, inp, pad_d=_pad_to_32_bytes(w), expect_kernel=f"gemm_{dtype}_tc<pair,direct")
    if _pairs_resident() == 76:
        assert lib.gemm_last_kernel() == f"gemm_{dtype}_tc<pair,direct,split-tail>"


# ------------------------------------------------ epilogue edge cases of the pair kernel
def test_direct_epilogue_narrow_n_one_partial_chunk():
    # 77 x 1 pair tiles of which only 24 columns exist: every chunk is the
    # partial edge chunk (guarded scalar stores), with and without C
    for beta in (0.0, -0.25):
        w = Workload("pair_narrow", 19712, 24, 64, 1.5, beta, "bf16", ROW, COL, ROW)
        inp = make_inputs(w, seed=47, ld_multiple=8)
        full_check(w, inp, pad_d=_pad_to_32_bytes(w), expect_kernel="gemm_bf16_tc<pair,direct")


def _with_ldc(w, inp, ldc):
    """inp with C (row-major) stored again at leading dimension ldc; A and B unchanged."""
    assert w.order_cd == ROW and ldc >= w.N
    C = torch.zeros((w.M, ldc), dtype=torch.float32)
    C[:, : w.N] = inp["C_logical"]
    return dict(inp, C=C, ldc=ldc)


@pytest.mark.parametrize("shape", [PAIR_SHAPE, (2000, 3300, 777)])
def test_in_place_c_equals_d_pair_staged(shape):
    # C = D with rows that do not start on 16 bytes (ldc = ldd = N + 3): the
    # wide staged epilogue reads C into a box and writes D from it, whole
    # tiles and split tail tiles
    M, N, K = shape
    w = Workload("inplace_staged", M, N, K, 0.5, 1.0, "bf16", ROW, COL, ROW)
    inp = _with_ldc(w, make_inputs(w, seed=48, ld_multiple=8), N + 3)
    Dbuf, _, name = run_gpu(w, inp, in_place=True)
    assert name.startswith("gemm_bf16_tc<pair") and "direct" not in name, name
    ref, S = oracle_full(w, inp)
    assert_within(w, logical_d(w, Dbuf), ref, S, c_logical(w, inp))


def test_c_rows_off_32_bytes_take_the_staged_epilogue():
    # D rows on 32 bytes but C rows only on 16 (ldc = N + 4): the direct
    # epilogue needs both, so the staged one (TMA C boxes) serves the call
    M, N, K = PAIR_SHAPE
    w = Workload("pair_c16", M, N, K, 1.5, -0.25, "bf16", ROW, COL, ROW)
    inp = _with_ldc(w, make_inputs(w, seed=49, ld_multiple=8), N + 4)  # rows on 16 bytes only
    assert inp["ldc"] % 8 == 4
    D, _, _ = full_check(w, inp, pad_d=_pad_to_32_bytes(w), expect_kernel="gemm_bf16_tc<pair")
    assert "direct" not in lib.gemm_last_kernel()
