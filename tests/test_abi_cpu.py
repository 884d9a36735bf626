"""The C-ABI library on a machine without a GPU: it loads, exports exactly
the entry points include/*.h declare, and rejects bad arguments before
touching CUDA (argument checks need no device)."""
import ctypes
import os
import re
import subprocess

import pytest

import dense_gemm_08_gb300 as lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in ("gemm.h", "gemm_probe.h")]


def declared_functions():
    names = []
    for header in HEADERS:
        text = open(header).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(
            r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", text,
            flags=re.M)
    return sorted(set(names))


def test_every_header_is_listed():
    on_disk = sorted(f for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h"))
    assert on_disk == sorted(os.path.basename(h) for h in HEADERS)


def test_header_declares_the_abi():
    assert declared_functions() == sorted(lib.EXPORTED)


def test_library_exports_every_declared_symbol():
    dll = lib.library()
    for name in declared_functions():
        assert hasattr(dll, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = sorted(line.split()[-1] for line in out.splitlines()
                      if " T " in line and not line.split()[-1].startswith("_"))
    assert exported == declared_functions()


def test_status_strings():
    for st in range(6):
        assert lib.gemm_status_string(st)
    assert lib.gemm_status_string(99) == "unknown status"


@pytest.mark.parametrize("fn_name", ["gemm_f32", "gemm_bf16_f32acc"])
def test_argument_errors_without_a_device(fn_name):
    fn = getattr(lib, fn_name)
    fake = 1 << 20  # never dereferenced: the checks run before any CUDA call
    good = dict(M=8, N=8, K=8, alpha=1.0, A=fake, lda=8, oa=0, B=fake, ldb=8, ob=0, beta=0.0,
                C=None, ldc=8, D=fake, ldd=8, ocd=0)
    bad = [dict(M=-1), dict(N=-3), dict(K=-1), dict(M=1 << 31), dict(oa=2), dict(ocd=5),
           dict(lda=7), dict(ldb=7), dict(ldd=7), dict(oa=1, lda=7), dict(ocd=1, ldd=7),
           dict(beta=1.0), dict(beta=1.0, C=fake, ldc=7), dict(A=None), dict(B=None),
           dict(D=None), dict(D=fake + 2), dict(A=fake + 1), dict(C=fake + 2, beta=1.0),
           # M * N above 2^43 (lda = K, ldb = ldd = N: leading dimensions valid)
           dict(M=1 << 22, N=(1 << 21) + 1, ldb=(1 << 21) + 1, ldd=(1 << 21) + 1)]
    for change in bad:
        a = dict(good, **change)
        st = fn(a["M"], a["N"], a["K"], a["alpha"], a["A"], a["lda"], a["oa"], a["B"], a["ldb"],
                a["ob"], a["beta"], a["C"], a["ldc"], a["D"], a["ldd"], a["ocd"], stream=0,
                check=False)
        assert st == lib.GEMM_ERR_INVALID_VALUE, change
    # M == 0 is a no-op even with NULL pointers
    assert fn(0, 8, 8, 1.0, None, 8, 0, None, 8, 0, 0.0, None, 8, None, 8, 0, stream=0) == 0
    assert lib.gemm_last_kernel() == ""


def test_probe_argument_errors_without_a_device():
    for cg, n in [(0, 10), (3, 10), (1, 0), (2, -5), (1, 1 << 41)]:
        st, _ = lib.gemm_probe_tc_bf16(cg, n, stream=0, check=False)
        assert st == lib.GEMM_ERR_INVALID_VALUE, (cg, n)
    for trips in [0, -1, 1 << 41]:
        st, _ = lib.gemm_probe_fma_f32(trips, stream=0, check=False)
        assert st == lib.GEMM_ERR_INVALID_VALUE, trips
    for t in [0, 999, 11 * 10 ** 9]:
        assert lib.gemm_probe_wait_timeout(t, stream=0, check=False) == lib.GEMM_ERR_INVALID_VALUE
    # a NULL flops pointer is refused
    assert lib.library().gemm_probe_fma_f32(10, None, None) == lib.GEMM_ERR_INVALID_VALUE
    assert lib.library().gemm_probe_tc_bf16(1, 10, None, None) == lib.GEMM_ERR_INVALID_VALUE


def test_valid_call_without_a_device_reports_unsupported_device():
    # all arguments valid: the library then needs an sm_103 device and says so
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    fake = 1 << 20
    st = lib.gemm_f32(8, 8, 8, 1.0, fake, 8, 0, fake, 8, 0, 0.0, None, 8, fake, 8, 0, stream=0,
                      check=False)
    assert st == lib.GEMM_ERR_UNSUPPORTED_DEVICE
