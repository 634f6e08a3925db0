"""Build libtq.so in-tree with nvcc for sm_103a (GB300).

Each translation unit is compiled in parallel, then linked into
``kv_cache_vector_head_gb300/libtq.so``.  Run ``python -m
kv_cache_vector_head_gb300.build`` or call :func:`build`.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libtq.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CUDA_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "-Xptxas", "-O3"]
SOURCES = ["tq_host.cpp", "tq_api.cu", "tq_quantize.cu", "tq_decode.cu"]


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found")
    return p


def _compile(src: str, verbose: bool, out_dir: str = OUT_DIR, defines=()) -> str:
    obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *CUDA_FLAGS, *defines, "-c", os.path.join(CSRC, src), "-o", obj]
    if src.endswith(".cpp"):
        cmd = [nvcc(), "-x", "c++", "-O2", "-std=c++17", "-Xcompiler", "-fPIC", "-c",
               os.path.join(CSRC, src), "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v") if src.endswith(".cu") else None
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"compile failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def _build(lib: str, out_dir: str, defines=(), verbose: bool = False, force: bool = False) -> str:
    os.makedirs(out_dir, exist_ok=True)
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    deps = srcs + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    deps.append(os.path.join(os.path.dirname(HERE), "include", "tq.h"))
    if not force and os.path.exists(lib):
        lib_t = os.path.getmtime(lib)
        if all(os.path.getmtime(d) <= lib_t for d in deps):
            return lib
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, out_dir, defines), SOURCES))
    tmp = lib + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build(verbose: bool = False, force: bool = False) -> str:
    """libtq.so, the library."""
    return _build(LIB, OUT_DIR, (), verbose, force)


TEST_HOOKS_LIB = os.path.join(HERE, "libtq_testhooks.so")


def build_test_hooks(verbose: bool = False, force: bool = False) -> str:
    """libtq_testhooks.so: the same sources built with TQ_TEST_HOOKS, for the test that makes a
    bounded device wait run out (short wait limit, tq_test_wait_fault).  Not used by the library."""
    return _build(TEST_HOOKS_LIB, os.path.join(HERE, "_build_hooks"), ("-DTQ_TEST_HOOKS",), verbose, force)


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
