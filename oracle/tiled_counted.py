"""Counted naive and tiled matrix products -- TEST INFRASTRUCTURE ONLY.

A restatement, in plain Python loops over small integer matrices, of the
traffic model in "Understanding roofline and tiling through matrix
multiplication" (tensor2silicon-lab, week 4):

* section 6.2 traces C = A @ B for 4 x 4 matrices with 2 x 2 output tiles and
  a K slice of width 2: per output tile the partial sums acc[T, T] are set to
  zero, each K step fetches a T x T slice of A and of B from "HBM" (2*T*T
  element reads), adds their product into acc (2*T^3 FLOPs, an FMA counting
  as 2), and only after the last K step is the tile of C written once (T*T
  element writes);
* section 6.3 gives that loop structure in words; section 10.2 describes the
  counting convention: copying a slice out of the source matrix counts as an
  HBM read, re-reading the copied slice counts as on-chip reuse;
* the "no reuse" baseline (section 6.2.4, 7.2) reads A_ik and B_kj from HBM
  for every multiply and writes each output once.

Element sizes are 4 bytes (FP32) as on that page.  These functions pin the
double-precision oracle (``oracle.gemm``) and the byte model the benchmark
uses: with small integers every sum is exact, so tiled == naive == oracle.
"""
from __future__ import annotations

from dataclasses import dataclass, field

ELEM_BYTES = 4  # FP32, as in the page's common example


@dataclass
class Counts:
    reads: int = 0   # element reads from HBM (A and B)
    writes: int = 0  # element writes to HBM (C)
    flops: int = 0   # an FMA counts as 2 FLOPs

    @property
    def hbm_bytes(self) -> int:
        return ELEM_BYTES * (self.reads + self.writes)

    @property
    def intensity(self) -> float:
        return self.flops / self.hbm_bytes


@dataclass
class StepRecord:
    """State of one output tile after one K step (for hand-trace checks)."""
    tile_row: int
    tile_col: int
    k0: int
    reads: int           # element reads of this step
    flops: int           # FLOPs of this step
    acc: list = field(default_factory=list)  # copy of acc[T][T] after the step


def _shape(a, b):
    n_i, n_k = len(a), len(a[0])
    assert len(b) == n_k
    n_j = len(b[0])
    return n_i, n_k, n_j


def naive_counted(a, b):
    """Every multiply fetches its two operands; each output is written once."""
    n_i, n_k, n_j = _shape(a, b)
    cnt = Counts()
    c = [[0] * n_j for _ in range(n_i)]
    for i in range(n_i):
        for j in range(n_j):
            acc = 0
            for k in range(n_k):
                acc += a[i][k] * b[k][j]
                cnt.reads += 2
                cnt.flops += 2
            c[i][j] = acc
            cnt.writes += 1
    return c, cnt


def tiled_counted(a, b, tile, trace=None):
    """Square output tiles of side ``tile`` and K slices of width ``tile``.

    ``tile`` must divide every dimension (the page's examples have no
    boundary padding).  If ``trace`` is a list, one StepRecord per (tile,
    K step) is appended to it.
    """
    n_i, n_k, n_j = _shape(a, b)
    T = tile
    assert n_i % T == 0 and n_k % T == 0 and n_j % T == 0, "tile must divide the shape"
    cnt = Counts()
    c = [[None] * n_j for _ in range(n_i)]
    for i0 in range(0, n_i, T):
        for j0 in range(0, n_j, T):
            acc = [[0] * T for _ in range(T)]  # kept across the whole K loop
            for k0 in range(0, n_k, T):
                # fetch the two slices: the only HBM reads of this step
                a_slice = [[a[i0 + i][k0 + k] for k in range(T)] for i in range(T)]
                b_slice = [[b[k0 + k][j0 + j] for j in range(T)] for k in range(T)]
                step_reads = 2 * T * T
                step_flops = 0
                for i in range(T):
                    for j in range(T):
                        for k in range(T):
                            acc[i][j] += a_slice[i][k] * b_slice[k][j]
                            step_flops += 2
                cnt.reads += step_reads
                cnt.flops += step_flops
                if trace is not None:
                    trace.append(StepRecord(i0 // T, j0 // T, k0, step_reads, step_flops,
                                            [row[:] for row in acc]))
            # the tile of C is written once, after the last K step
            for i in range(T):
                for j in range(T):
                    c[i0 + i][j0 + j] = acc[i][j]
            cnt.writes += T * T
    return c, cnt


def tiled_traffic_bytes(n: int, tile: int) -> int:
    """Closed form of the tiled model for an n x n x n FP32 product.

    (n/T)^2 output tiles, n/T K steps each, 2*T^2 four-byte reads per step,
    plus one write of C: Q_T = 8 n^3 / T + 4 n^2 (section 8.1).  ``tile=1``
    is the no-reuse case, Q = 8 n^3 + 4 n^2 (section 7.2).
    """
    assert n % tile == 0
    return 8 * n ** 3 // tile + 4 * n ** 2
