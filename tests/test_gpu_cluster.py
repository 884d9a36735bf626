"""GPU parity of the FP32 cluster kernel (few 64 x 64 tiles; each tile's K
range split over the 2, 4 or 8 CTAs of a cluster, partial tiles added
through distributed shared memory in rank order).

Covers every storage order, each cluster size, ragged M, N and K edges,
slices that are partly or wholly past K, padded leading dimensions, the
in-place update C == D, exactness and run-to-run identity on small integers,
and the size limits past which the tiled kernel takes over."""
import itertools

import numpy as np
import pytest
import torch

import dense_gemm_08_gb300 as lib
from dense_gemm_08_gb300.inputs import ROW, Workload, make_inputs
from gemm_harness import (assert_within, c_logical, check_canary, logical_d, oracle_full,
                          run_gpu)

pytestmark = pytest.mark.gpu

ORDERS = list(itertools.product((0, 1), repeat=3))


def check(w, inp, pad_d=0, expect=None, in_place=False):
    Dbuf, _, name = run_gpu(w, inp, pad_d=pad_d, in_place=in_place)
    if expect is not None:
        assert name.startswith(expect), name
    ref, S = oracle_full(w, inp)
    assert_within(w, logical_d(w, Dbuf), ref, S, c_logical(w, inp), str((w.M, w.N, w.K)))
    if pad_d:
        check_canary(w, Dbuf)
    return Dbuf, name


# (M, N, K) -> cluster size on a 152-SM GB300
SHAPES = [((256, 256, 256), 8),    # 16 tiles, slices of 32
          ((65, 129, 333), 8),     # ragged; slices of 64, the last two past K
          ((300, 600, 200), 2),    # 50 tiles: only pairs fit one CTA per SM
          ((130, 140, 150), 4),    # 9 tiles; K too short for 8 slices of 32
          ((9, 70, 64), 2),        # two tiles, one K chunk per CTA
          ((256, 256, 1024), 8)]   # the longest K it takes (8 slices of 128)


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("orders", ORDERS)
@pytest.mark.parametrize("shape,cl", SHAPES)
def test_every_order_and_cluster_size_full(shape, cl, orders):
    M, N, K = shape
    w = Workload("cluster", M, N, K, 1.5, -0.25, "f32", *orders)
    inp = make_inputs(w, seed=M + 7 * N + 13 * K, pad=3)
    expect = f"sgemm_cluster<f32,ks:{cl}>" if _sms() == 152 else "sgemm_"
    check(w, inp, pad_d=3, expect=expect)


def test_in_place_update():
    w = Workload("cluster_inplace", 256, 192, 200, 0.5, 2.0, "f32", ROW, ROW, ROW)
    inp = make_inputs(w, seed=5)
    check(w, inp, in_place=True, expect="sgemm_cluster<f32")


@pytest.mark.parametrize("shape", [(256, 256, 256), (65, 129, 333)])
def test_small_integers_exact_and_repeatable(shape):
    M, N, K = shape
    w = Workload("cluster_int", M, N, K, 1.0, 0.0, "f32", ROW, ROW, ROW, dist="int")
    inp = make_inputs(w, seed=9)
    D1, name = check(w, inp, expect="sgemm_cluster<f32")
    ref, _ = oracle_full(w, inp)
    assert np.array_equal(logical_d(w, D1), ref.astype(np.float32))
    w2 = w.with_(dist="normal", alpha=1.5, beta=-0.25)
    inp2 = make_inputs(w2, seed=10)
    Da, _, _ = run_gpu(w2, inp2)
    Db, _, _ = run_gpu(w2, inp2)
    assert torch.equal(Da, Db)


@pytest.mark.parametrize("shape", [(256, 256, 1025),   # K beyond 8 slices of 128
                                   (700, 500, 100),    # 88 tiles: no cluster of 2 fits
                                   (256, 256, 63)])    # K too short to split
def test_outside_its_range_the_tiled_kernel_runs(shape):
    M, N, K = shape
    w = Workload("cluster_out", M, N, K, 1.5, -0.25, "f32", ROW, ROW, ROW)
    inp = make_inputs(w, seed=11)
    _, name = check(w, inp)
    assert name.startswith("sgemm_simt<f32"), name
