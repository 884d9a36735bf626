"""GPU tests of the split kernels' per-stream counters.

Kernels that split a tile's K range over CTAs that are not one cluster (the
CTA-pair kernel's split last round, the CUDA-core stream-K tail, the small-M
kernel's K slices) count the finished pieces in counters that belong to the
stream and persist between calls; the piece that completes a count returns
it to zero, so no call clears them (a captured call takes fresh zeroed
counters instead).  The single-CTA tensor-core split-K adds its pieces
inside a thread-block cluster and takes no counters; it runs beside the
others here.  These tests check that calls of every variant -- back to back
in any order, on two streams at once, after a kernel gave up a bounded wait,
and replayed from a captured graph beside eager calls -- give the same bits
as a first call that is checked against the oracle.  Calls may come from any
number of host threads, on one stream or on several (cudaStreamPerThread
included); counters a stream outgrows are freed in stream order."""
import numpy as np
import pytest
import torch

import dense_gemm_08_gb300 as lib
from dense_gemm_08_gb300.inputs import COL, ROW, Workload, make_inputs, output_buffer
from gemm_harness import assert_within, oracle_points, sample_points

pytestmark = pytest.mark.gpu

# (workload, expected kernel prefix)
CASES = [
    (Workload("tc_splitk", 300, 600, 2048, 1.5, -0.25, "bf16", ROW, COL, ROW), "gemm_bf16_tc<splitk,"),
    (Workload("pair_tail", 2304, 2560, 1024, 0.5, 1.0, "bf16", ROW, COL, ROW), "gemm_bf16_tc<pair"),
    (Workload("f16_splitk", 300, 600, 2048, 1.0, 0.5, "f16", COL, ROW, COL), "gemm_f16_tc<splitk,"),
    (Workload("simt_splitk", 384, 384, 1000, 1.5, -0.25, "f32", ROW, ROW, ROW), "sgemm_simt<f32"),
    (Workload("simt_tail", 2560, 2048, 512, 1.0, 0.0, "f32", ROW, COL, ROW), "sgemm_simt<f32"),
    (Workload("skinny", 4, 3000, 5000, 1.5, -0.25, "f32", ROW, ROW, ROW), "skinny<f32"),
]

FN = {"f32": lib.gemm_f32, "bf16": lib.gemm_bf16_f32acc, "f16": lib.gemm_f16_f32acc}


class Case:
    """Device copies of one workload's inputs, and a launcher into fresh D buffers."""

    def __init__(self, w, prefix, seed):
        self.w, self.prefix = w, prefix
        self.inp = make_inputs(w, seed=seed, ld_multiple=8)
        self.A = self.inp["A"].cuda()
        self.B = self.inp["B"].cuda()
        self.C = self.inp["C"].cuda() if self.inp["C"] is not None else None

    def launch(self, stream=None):
        D, ldd = output_buffer(self.w, device="cuda", fill=0.0)
        w, inp = self.w, self.inp
        FN[w.dtype](w.M, w.N, w.K, w.alpha, self.A, inp["lda"], w.order_a, self.B, inp["ldb"],
                    w.order_b, w.beta, self.C, inp["ldc"], D, ldd, w.order_cd, stream)
        assert lib.gemm_last_kernel().startswith(self.prefix), lib.gemm_last_kernel()
        return D

    def check_against_oracle(self, D):
        w = self.w
        Dl = D.cpu().numpy() if w.order_cd == ROW else D.cpu().numpy().T
        I, J = sample_points(w.M, w.N, np.random.default_rng(5), n_random=1500)
        ref, S = oracle_points(w, self.inp, I, J)
        C = self.inp["C_logical"].numpy()[I, J] if self.inp["C_logical"] is not None else None
        assert_within(w, Dl[I, J], ref, S, C, "first call")


@pytest.fixture(scope="module")
def cases():
    out = [Case(w, prefix, seed=40 + i) for i, (w, prefix) in enumerate(CASES)]
    torch.cuda.synchronize()
    return out


def _first_results(cases):
    first = [c.launch() for c in cases]
    torch.cuda.synchronize()
    assert lib.gemm_last_device_status() == lib.GEMM_OK
    return first


def test_back_to_back_calls_of_every_split_variant(cases):
    first = _first_results(cases)
    for c, D in zip(cases, first):
        c.check_against_oracle(D)
    order = np.random.default_rng(3).permutation(np.repeat(np.arange(len(cases)), 4))
    got = [(i, cases[i].launch()) for i in order]  # no synchronisation in between
    torch.cuda.synchronize()
    assert lib.gemm_last_device_status() == lib.GEMM_OK
    for i, D in got:
        assert torch.equal(D, first[i]), cases[i].w.name


def test_two_streams_at_once(cases):
    first = _first_results(cases)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for s in (s1, s2):
        s.wait_stream(torch.cuda.current_stream())
    got = []
    for rep in range(3):
        for i in range(len(cases)):
            j = (i + 1 + rep) % len(cases)
            with torch.cuda.stream(s1):
                got.append((i, cases[i].launch(s1)))
            with torch.cuda.stream(s2):
                got.append((j, cases[j].launch(s2)))
    torch.cuda.synchronize()
    assert lib.gemm_last_device_status() == lib.GEMM_OK
    for i, D in got:
        assert torch.equal(D, first[i]), cases[i].w.name


def test_split_variants_after_a_wait_gave_up(cases):
    first = _first_results(cases)
    assert lib.gemm_probe_wait_timeout(2_000_000) == lib.GEMM_OK
    # reading the timeout also returns every split counter on the device to zero
    assert lib.gemm_last_device_status() == lib.GEMM_ERR_TIMEOUT
    got = [(i, c.launch()) for i, c in enumerate(cases)]
    torch.cuda.synchronize()
    assert lib.gemm_last_device_status() == lib.GEMM_OK
    for i, D in got:
        assert torch.equal(D, first[i]), cases[i].w.name


def test_captured_graph_replays_beside_eager_calls(cases):
    """A graph captured with every split variant gets its own zeroed counters
    per captured launch, so replaying it -- here on a side stream while eager
    calls of the same variants run on the default stream -- gives the same
    bits as eager calls, replay after replay."""
    first = _first_results(cases)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        captured = [c.launch() for c in cases]
    side = torch.cuda.Stream()
    for _ in range(3):
        for D in captured:
            D.zero_()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            graph.replay()
        eager = [c.launch() for c in cases]
        torch.cuda.synchronize()
        assert lib.gemm_last_device_status() == lib.GEMM_OK
        for i, D in enumerate(captured):
            assert torch.equal(D, first[i]), cases[i].w.name
        for i, D in enumerate(eager):
            assert torch.equal(D, first[i]), cases[i].w.name


def test_host_threads_on_their_own_streams(cases):
    """Four host threads, each on its own stream, call every split variant at
    the same time (the binding releases the GIL during a call): each stream
    has its own counters, so every result matches the first call."""
    import threading
    first = _first_results(cases)
    got, errors = {}, []

    def worker(t):
        try:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            out = []
            with torch.cuda.stream(s):
                for rep in range(3):
                    for i in range(len(cases)):
                        j = (i + t + rep) % len(cases)
                        out.append((j, cases[j].launch(s)))
            s.synchronize()
            got[t] = out
        except Exception as e:  # surfaced below, in the test's thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    torch.cuda.synchronize()
    assert lib.gemm_last_device_status() == lib.GEMM_OK
    for t, out in got.items():
        for i, D in out:
            assert torch.equal(D, first[i]), (t, cases[i].w.name)


def test_host_threads_on_one_stream(cases):
    """Two host threads call every split variant on the SAME stream at once:
    a call holds the stream's counters until its kernel is enqueued, so the
    launches of the stream are enqueued one after another and every result
    is bit-identical to the oracle-checked first call."""
    import threading
    first = _first_results(cases)
    for c, D in zip(cases, first):
        c.check_against_oracle(D)
    shared = torch.cuda.Stream()
    shared.wait_stream(torch.cuda.current_stream())
    got, errors = {}, []
    barrier = threading.Barrier(2)

    def worker(t):
        try:
            out = []
            barrier.wait()
            with torch.cuda.stream(shared):
                for rep in range(4):
                    for i in range(len(cases)):
                        j = (i + 3 * t + rep) % len(cases)
                        out.append((j, cases[j].launch(shared)))
            got[t] = out
        except Exception as e:  # surfaced below, in the test's thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    torch.cuda.synchronize()
    assert lib.gemm_last_device_status() == lib.GEMM_OK
    assert sorted(got) == [0, 1]
    for t, out in got.items():
        for i, D in out:
            assert torch.equal(D, first[i]), (t, cases[i].w.name)


def test_per_thread_default_stream_in_two_threads(cases):
    """cudaStreamPerThread is one handle value but a different stream in each
    host thread; the library tells the streams apart by their unique id, so
    two threads calling the split variants on it at once keep separate
    counters and get the first call's bits."""
    import threading
    per_thread = 2  # cudaStreamPerThread
    first = _first_results(cases)
    got, errors = {}, []
    barrier = threading.Barrier(2)

    def worker(t):
        try:
            out = []
            barrier.wait()
            for rep in range(4):
                for i in range(len(cases)):
                    j = (i + t + rep) % len(cases)
                    out.append((j, cases[j].launch(per_thread)))
            torch.cuda.synchronize()
            got[t] = out
        except Exception as e:  # surfaced below, in the test's thread
            errors.append(repr(e))

    torch.cuda.synchronize()
    threads = [threading.Thread(target=worker, args=(t,)) for t in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    torch.cuda.synchronize()
    assert lib.gemm_last_device_status() == lib.GEMM_OK
    for t, out in got.items():
        for i, D in out:
            assert torch.equal(D, first[i]), (t, cases[i].w.name)


def test_outgrown_counters_are_freed():
    """Eleven calls on one stream, each splitting more column blocks than the
    last, grow the stream's counters ten times; each outgrown buffer is freed
    in stream order, so afterwards the stream holds one buffer (the last
    size) and the pool has nothing else in use.  gemm_release_memory frees
    even that, and the next call starts from fresh counters.  Every result is
    checked against the oracle."""
    lib.gemm_release_memory()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    sizes = []
    # the small-M kernel on row-major B: one counter per 128-column block,
    # t blocks (K = 2048 is cut into at least two slices for every t here)
    for t in (1, 17, 33, 49, 65, 81, 97, 113, 129, 145, 161):
        w = Workload(f"grow_{t}", 4, 128 * t, 2048, 1.0, 0.0, "f32", ROW, ROW, ROW)
        c = Case(w, "skinny<f32", seed=t)
        D = c.launch(s)
        s.synchronize()
        c.check_against_oracle(D)
        info = lib.gemm_memory_info()
        assert info["split_streams"] == 1, info
        sizes.append(info["split_bytes"])
    assert all(b > a for a, b in zip(sizes, sizes[1:])), sizes  # ten growths
    # the last call's 161 counters, rounded up to 16 words
    assert sizes[-1] == 176 * 4, sizes
    assert lib.gemm_release_memory() == lib.GEMM_OK
    info = lib.gemm_memory_info()
    assert info["split_streams"] == 0 and info["split_bytes"] == 0, info
    assert info["pool_used_bytes"] == 0 and info["pool_reserved_bytes"] == 0, info
    w = Workload("after_release", 4, 3000, 5000, 1.5, -0.25, "f32", ROW, ROW, ROW)
    c = Case(w, "skinny<f32", seed=99)
    D = c.launch(s)
    s.synchronize()
    c.check_against_oracle(D)
    assert lib.gemm_last_device_status() == lib.GEMM_OK


def test_cluster_split_takes_no_memory():
    """The single-CTA tensor-core split-K adds its K pieces in the shared
    memory of one thread-block cluster: calls of it, eager and captured,
    leave the library's pool and the stream's counters untouched."""
    assert lib.gemm_release_memory() == lib.GEMM_OK
    cases = [Case(w, prefix, seed=60 + i) for i, (w, prefix) in enumerate(CASES)
             if prefix.startswith("gemm_") and "splitk" in prefix]
    assert len(cases) == 2
    first = [c.launch() for c in cases]
    torch.cuda.synchronize()
    for c, D in zip(cases, first):
        c.check_against_oracle(D)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        captured = [c.launch() for c in cases]
    graph.replay()
    torch.cuda.synchronize()
    for D, ref in zip(captured, first):
        assert torch.equal(D, ref)
    info = lib.gemm_memory_info()
    assert info["split_streams"] == 0 and info["split_bytes"] == 0, info
    assert info["pool_used_bytes"] == 0 and info["pool_reserved_bytes"] == 0, info
    assert lib.gemm_last_device_status() == lib.GEMM_OK
