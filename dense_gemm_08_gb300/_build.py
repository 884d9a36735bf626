"""Builds the CUDA library libdense_gemm_08_gb300.so in-tree with nvcc.

One -gencode (sm_103a), translation units compiled in parallel, static
CUDA runtime, only the C ABI of include/gemm.h exported.  The ptxas
resource report (registers, spills, shared memory per kernel) of each unit
is kept in _build/ptxas_<unit>.log.
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_NAME = "libdense_gemm_08_gb300.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)

SOURCES = ["gemm_api.cu", "sgemm_simt.cu", "sgemm_cluster.cu", "gemm_tc.cu", "workspace.cu",
           "probe.cu", "skinny.cu"]
HEADERS = [os.path.join(CSRC, "internal.h"), os.path.join(CSRC, "epilogue.cuh"),
           os.path.join(INCLUDE, "gemm.h"), os.path.join(INCLUDE, "gemm_probe.h")]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC,-fvisibility=hidden",
    "-Xptxas", "-v",
    "-I" + INCLUDE,
]


def _nvcc() -> str:
    cuda_home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(cuda_home, "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if needed) and return the path of the shared library."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = _nvcc()
    objs, procs = [], []
    for src in SOURCES:
        src_path = os.path.join(CSRC, src)
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        objs.append(obj)
        if force or _stale(obj, [src_path, *HEADERS]):
            log = open(os.path.join(BUILD_DIR, "ptxas_" + src.replace(".cu", ".log")), "w")
            cmd = [nvcc, *NVCC_FLAGS, "-c", src_path, "-o", obj]
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            procs.append((src, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT), log))
    failed = []
    for src, proc, log in procs:
        proc.wait()
        log.close()
        if proc.returncode != 0:
            failed.append(src)
    if failed:
        msgs = []
        for src in failed:
            with open(os.path.join(BUILD_DIR, "ptxas_" + src.replace(".cu", ".log"))) as f:
                msgs.append(f"--- {src}\n" + f.read()[-4000:])
        raise RuntimeError("nvcc failed:\n" + "\n".join(msgs))
    if force or _stale(LIB_PATH, objs):
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        cmd = [nvcc, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-o", tmp, *objs]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


def build_variant(tag: str, defines: dict, units=("gemm_tc.cu",), verbose: bool = False) -> str:
    """A second build of the library with preprocessor `defines` applied to
    `units` (the other translation units are the default build's objects),
    in _build/<tag>/; returns its path.  For measurements that compare a
    compile-time choice (e.g. the ring depth) in otherwise the same library."""
    build(verbose=verbose)
    out_dir = os.path.join(BUILD_DIR, tag)
    os.makedirs(out_dir, exist_ok=True)
    flags = [f"-D{k}={v}" for k, v in sorted(defines.items())]
    nvcc = _nvcc()
    objs = []
    for src in SOURCES:
        if src not in units:
            objs.append(os.path.join(BUILD_DIR, src.replace(".cu", ".o")))
            continue
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        with open(os.path.join(out_dir, "ptxas_" + src.replace(".cu", ".log")), "w") as log:
            subprocess.run([nvcc, *NVCC_FLAGS, *flags, "-c", os.path.join(CSRC, src), "-o", obj],
                           stdout=log, stderr=subprocess.STDOUT, check=True)
    lib = os.path.join(out_dir, LIB_NAME)
    subprocess.run([nvcc, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-o", lib,
                    *objs], check=True)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
