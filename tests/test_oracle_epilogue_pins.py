"""Pins of the oracle's fused epilogue (bias, ReLU, GELU) -- no GPU.

Each property below is fixed by the mathematics, not by retyping the oracle:
ReLU(x) - ReLU(-x) = x and ReLU(x) + ReLU(-x) = |x|; for the tanh form of
GELU, g(x) - g(-x) = x (tanh is odd), g(0) = 0, g(x) -> x and g(-x) -> 0
for large x, and g stays within the approximation's published error of the
exact GELU x * Phi(x) (Phi from math.erf); the bias is added along columns.
Planted mistakes in a copy of the oracle must fail these checks.
"""
import ctypes
import math
import os
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _epi(D, bias=None, act=oracle.ACT_NONE, lib=None):
    D = np.ascontiguousarray(D, dtype=np.float64).copy()
    if lib is None:
        return oracle.epilogue(D, bias, act)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    rc = lib.oracle_epilogue(D.shape[0], D.shape[1], D.ctypes.data,
                             None if b is None else b.ctypes.data, act)
    assert rc == 0
    return D


def check_relu(lib=None):
    rng = np.random.default_rng(1)
    x = rng.normal(size=(7, 9))
    pos = _epi(x, act=oracle.ACT_RELU, lib=lib)
    neg = _epi(-x, act=oracle.ACT_RELU, lib=lib)
    return np.array_equal(pos - neg, x) and np.array_equal(pos + neg, np.abs(x)) and (pos >= 0).all()


def check_gelu(lib=None):
    rng = np.random.default_rng(2)
    x = rng.normal(scale=3.0, size=(6, 11))
    g = _epi(x, act=oracle.ACT_GELU, lib=lib)
    gm = _epi(-x, act=oracle.ACT_GELU, lib=lib)
    ok = np.allclose(g - gm, x, rtol=0, atol=1e-14)
    special = _epi(np.array([[0.0, 10.0, -10.0, 30.0]]), act=oracle.ACT_GELU, lib=lib)[0]
    ok &= special[0] == 0.0 and special[1] == 10.0 and abs(special[2]) < 1e-20 and special[3] == 30.0
    # the tanh form stays within 5e-4 of the exact GELU x * Phi(x)
    xs = np.linspace(-6, 6, 241).reshape(1, -1)
    gt = _epi(xs, act=oracle.ACT_GELU, lib=lib)[0]
    exact = np.array([v * 0.5 * (1.0 + math.erf(v / math.sqrt(2.0))) for v in xs[0]])
    ok &= float(np.max(np.abs(gt - exact))) < 5e-4
    # and at x = 1 the two differ by about 1.5e-4, not by 0
    ok &= 1e-5 < abs(gt[120 + 20] - exact[120 + 20]) < 5e-4
    return bool(ok)


def check_bias(lib=None):
    rng = np.random.default_rng(3)
    D = rng.integers(-5, 6, size=(5, 8)).astype(np.float64)
    bias = np.arange(8, dtype=np.float32) * 10.0  # distinct per column
    out = _epi(D, bias, oracle.ACT_NONE, lib=lib)
    return bool(np.array_equal(out - D, np.broadcast_to(bias.astype(np.float64), D.shape)))


def test_relu_identities():
    assert check_relu()


def test_gelu_tanh_form_properties():
    assert check_gelu()


def test_bias_goes_along_columns():
    assert check_bias()


def test_rejects_unknown_activation():
    with pytest.raises(ValueError):
        oracle.epilogue(np.zeros((2, 2)), None, 7)


MUTANTS = {
    "GELU cubic coefficient": ("0.044715 * x * x * x", "0.04715 * x * x * x", check_gelu),
    "GELU half dropped": ("x = 0.5 * x * (1.0 + tanh(", "x = x * (1.0 + tanh(", check_gelu),
    "bias along rows": ("x += (double)bias[j];", "x += (double)bias[i];", check_bias),
    "ReLU keeps negatives": ("x = x > 0.0 ? x : 0.0;", "x = x > -1.0 ? x : 0.0;", check_relu),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_epilogue_pins_catch_planted_mistakes(name, tmp_path):
    src = open(os.path.join(ROOT, "oracle", "gemm_oracle.c")).read()
    old, new, check = MUTANTS[name]
    assert src.count(old) == 1
    cfile = tmp_path / "mutant.c"
    cfile.write_text(src.replace(old, new))
    lib_path = tmp_path / "libmutant.so"
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", str(lib_path), str(cfile), "-lm"], check=True)
    lib = ctypes.CDLL(str(lib_path))
    lib.oracle_epilogue.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                    ctypes.c_void_p, ctypes.c_int]
    lib.oracle_epilogue.restype = ctypes.c_int
    assert not check(lib), f"mutant '{name}' survived"
