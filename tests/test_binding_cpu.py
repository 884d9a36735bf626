"""The Python binding's argument handling on the CPU: storage order and
leading dimension read from torch strides, and the gemm() helper's checks
that run before any call into the library."""
import pytest
import torch

import dense_gemm_08_gb300 as lib


def test_row_major_views():
    x = torch.zeros(3, 4)
    assert lib.storage_order(x) == (lib.ROW_MAJOR, 4)
    padded = torch.zeros(3, 8)[:, :5]  # rows 8 apart
    assert lib.storage_order(padded) == (lib.ROW_MAJOR, 8)


def test_column_major_views():
    x = torch.zeros(4, 3).t()  # 3 x 4, column-major, ld 3
    assert x.shape == (3, 4)
    assert lib.storage_order(x) == (lib.COL_MAJOR, 3)
    padded = torch.zeros(6, 3)[:5].t()  # 3 x 5, columns 3 apart
    assert lib.storage_order(padded) == (lib.COL_MAJOR, 3)


def test_single_rows_and_columns():
    assert lib.storage_order(torch.zeros(1, 5)) == (lib.ROW_MAJOR, 5)
    assert lib.storage_order(torch.zeros(5, 1))[0] in (lib.ROW_MAJOR, lib.COL_MAJOR)
    order, ld = lib.storage_order(torch.zeros(5, 1))
    assert ld >= (1 if order == lib.ROW_MAJOR else 5)


def test_rejects_other_layouts():
    with pytest.raises(ValueError):
        lib.storage_order(torch.zeros(4, 6)[:, ::2])  # columns 2 apart
    with pytest.raises(ValueError):
        lib.storage_order(torch.zeros(2, 3, 4))


def test_gemm_helper_checks_before_calling_the_library():
    a = torch.zeros(3, 4)
    with pytest.raises(ValueError):
        lib.gemm(a, torch.zeros(5, 2))  # inner dimensions differ
    with pytest.raises(TypeError):
        lib.gemm(a, torch.zeros(4, 2, dtype=torch.bfloat16))  # dtypes differ
    with pytest.raises(ValueError):
        lib.gemm(a, torch.zeros(4, 2), beta=1.0)  # beta != 0 without C
    with pytest.raises(ValueError):
        c = torch.zeros(2, 3).t()  # column-major C, row-major output
        lib.gemm(a, torch.zeros(4, 2), C=c, beta=1.0, out=torch.zeros(3, 2))
    with pytest.raises(TypeError):
        lib.gemm(a.to(torch.int32), torch.zeros(4, 2, dtype=torch.int32))
