"""Seeded synthetic inputs for the GEMM workloads.

Data only -- this module holds none of the GEMM's arithmetic.  Tests,
``bench.py`` and the smoke check draw every operand from here, so the CUDA
library and the CPU oracle always see the same bits.

Recipe (one ``torch.Generator('cpu')`` per call, seeded; draw order A, B, C):
  * the LOGICAL matrices are drawn row-major: A (M x K), then B (K x N), then
    C (M x N, only when beta != 0);
  * "uniform": ``torch.rand * 2 - 1`` in FP32 (uniform on [-1, 1));
    "normal": ``torch.randn * sigma`` in FP32; "int": ``torch.randint(-4, 5)``
    as FP32 (small integers in [-4, 4]);
  * BF16 / FP16 operands are the FP32 draws rounded to nearest-even
    (``Tensor.to(torch.bfloat16 / torch.float16)`` on the CPU); C stays FP32;
  * each operand is then laid out in its storage order with leading
    dimension = minimal + ``pad`` (column-major = the transpose stored
    row-major).
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch

ROW = 0
COL = 1


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    alpha: float
    beta: float
    dtype: str               # "f32" (gemm_f32), "bf16" (gemm_bf16_f32acc), "f16" (gemm_f16_f32acc)
    order_a: int = ROW
    order_b: int = ROW
    order_cd: int = ROW
    dist: str = "uniform"    # distribution of A and B: uniform | normal | int
    sigma: float = 1.0       # standard deviation for "normal"
    c_dist: str = "uniform"  # distribution of C (when beta != 0)
    c_sigma: float = 1.0

    @property
    def flops(self) -> int:
        """2MNK ("GEMM on NVIDIA GPUs", section 1; alpha/beta not counted)."""
        return 2 * self.M * self.N * self.K

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


ODD_SHAPES = [(4095, 4097, 1000), (127, 8191, 4096), (16384, 64, 8192), (1, 4096, 4096)]


def _odd(M, N, K, dtype):
    ob = COL if dtype == "bf16" else ROW
    return Workload(f"odd_{dtype}_{M}x{N}x{K}", M, N, K, 1.5, -0.25, dtype, ROW, ob, ROW,
                    "uniform", 1.0, "uniform")


WORKLOADS = {
    # FP32 256^3, row-major, alpha=1 beta=0, uniform[-1,1] (+ small-integer variant)
    "f32_256": Workload("f32_256", 256, 256, 256, 1.0, 0.0, "f32"),
    "f32_256_int": Workload("f32_256_int", 256, 256, 256, 1.0, 0.0, "f32", dist="int"),
    # FP32 4096^3, row-major, alpha=1 beta=0, uniform[-1,1]
    "f32_4096": Workload("f32_4096", 4096, 4096, 4096, 1.0, 0.0, "f32"),
    # BF16 8192^3, A row-major, B column-major, D FP32 row-major, N(0,1) -> bf16
    "bf16_8192": Workload("bf16_8192", 8192, 8192, 8192, 1.0, 0.0, "bf16", ROW, COL, ROW,
                          "normal", 1.0),
    # MLP up-projection: M=8192 tokens, K=4096, N=14336, alpha=0.5 beta=1,
    # A,B N(0,0.02) -> bf16, C N(0,1) FP32
    "bf16_mlp": Workload("bf16_mlp", 8192, 14336, 4096, 0.5, 1.0, "bf16", ROW, COL, ROW,
                         "normal", 0.02, "normal", 1.0),
    # FP16-input FP32-accumulate at 8192^3 (the Ada pipeline-depth study's
    # FP16 -> FP32 workload), A row-major, B column-major, N(0,1) -> FP16
    "f16_8192": Workload("f16_8192", 8192, 8192, 8192, 1.0, 0.0, "f16", ROW, COL, ROW,
                         "normal", 1.0),
}
for _M, _N, _K in ODD_SHAPES:
    for _dt in ("f32", "bf16"):
        _w = _odd(_M, _N, _K, _dt)
        WORKLOADS[_w.name] = _w


def _draw(g, shape, dist, sigma):
    if dist == "uniform":
        return torch.rand(shape, generator=g, dtype=torch.float32) * 2 - 1
    if dist == "normal":
        return torch.randn(shape, generator=g, dtype=torch.float32) * sigma
    if dist == "int":
        return torch.randint(-4, 5, shape, generator=g).to(torch.float32)
    raise ValueError(dist)


def _lay_out(x, order, pad, ld_multiple=1):
    """Storage buffer (contiguous 2-D) and leading dimension of logical x in `order`."""
    if order == COL:
        x = x.t()
    rows, cols = x.shape
    ld = max(cols + pad, 1)
    ld = -(-ld // ld_multiple) * ld_multiple
    buf = torch.zeros((max(rows, 1), ld), dtype=x.dtype)
    buf[:rows, :cols] = x
    return buf, ld


def make_inputs(w: Workload, seed: int = 0, pad: int = 0, ld_multiple: int = 1):
    """CPU tensors for workload `w`.

    Returns a dict with
      A, B: storage buffers (float32, or bfloat16 for w.dtype == "bf16"),
      lda, ldb: their leading dimensions,
      C: float32 storage buffer in w.order_cd (None when beta == 0), ldc,
      A_logical, B_logical, C_logical: the logical matrices (same values).
    Leading dimensions are minimal + pad, rounded up to a multiple of ld_multiple.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    a = _draw(g, (w.M, w.K), w.dist, w.sigma)
    b = _draw(g, (w.K, w.N), w.dist, w.sigma)
    c = _draw(g, (w.M, w.N), w.c_dist, w.c_sigma) if w.beta != 0 else None
    if w.dtype in ("bf16", "f16"):
        t = torch.bfloat16 if w.dtype == "bf16" else torch.float16
        a = a.to(t)
        b = b.to(t)
    A, lda = _lay_out(a, w.order_a, pad, ld_multiple)
    B, ldb = _lay_out(b, w.order_b, pad, ld_multiple)
    if c is not None:
        C, ldc = _lay_out(c, w.order_cd, pad, ld_multiple)
    else:
        C, ldc = None, max(w.N if w.order_cd == ROW else w.M, 1) + pad
    return dict(A=A, lda=lda, B=B, ldb=ldb, C=C, ldc=ldc, A_logical=a, B_logical=b,
                C_logical=c)


def output_buffer(w: Workload, pad: int = 0, device="cpu", fill=float("nan"), pad_rows: int = 0):
    """Storage for D in w.order_cd, pre-filled: leading dimension minimal + pad,
    and pad_rows spare rows (of the storage) after the matrix."""
    rows, cols = (w.M, w.N) if w.order_cd == ROW else (w.N, w.M)
    ld = max(cols + pad, 1)
    shape = (max(rows, 1) + pad_rows, ld)
    return torch.full(shape, fill, dtype=torch.float32, device=device), ld
