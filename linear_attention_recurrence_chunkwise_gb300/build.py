"""Build libkda.so in-tree with nvcc for sm_103a.

Each translation unit under ``csrc/`` compiles in parallel to an object in
``_build/``; the objects link into ``libkda.so`` beside this file against the
shared CUDA runtime (so the library and PyTorch share one runtime).  Only
stale objects are rebuilt.  ``build(bounds_check=True)`` makes the
bounds-checked variant ``libkda_bounds.so`` (objects in ``_build_bounds/``),
whose kernels check every computed global index and report KDA_ERR_BOUNDS;
``build(timeout_probe=True)`` makes the test-only ``libkda_timeout.so``, in
which one wait of the tensor-core prefill runs out after 2 ms (the tests of
the timeout path use it).
Run ``python -m linear_attention_recurrence_chunkwise_gb300.build``.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libkda.so")
BUILD_BOUNDS = os.path.join(PKG, "_build_bounds")
LIB_BOUNDS = os.path.join(PKG, "libkda_bounds.so")
BUILD_TIMEOUT = os.path.join(PKG, "_build_timeout")
LIB_TIMEOUT = os.path.join(PKG, "libkda_timeout.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def _flags(verbose_ptxas: bool, bounds_check: bool = False, timeout_probe: bool = False):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    if bounds_check:
        f += ["-DKDA_BOUNDS_CHECK=1"]
    if timeout_probe:
        # test-only: a 2 ms wait limit and one mbarrier arrive left out, so a
        # wait of the tensor-core prefill runs out of time (the timeout path)
        f += ["-DKDA_WAIT_LIMIT_NS=2000000ull", "-DKDA_TEST_SKIP_ARRIVE=1"]
    return f


def _deps_mtime() -> float:
    hdrs = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))
    return max([os.path.getmtime(h) for h in hdrs] + [0.0])


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None,
          bounds_check: bool = False, timeout_probe: bool = False) -> str:
    build_dir, lib_path = (BUILD_BOUNDS, LIB_BOUNDS) if bounds_check else \
        (BUILD_TIMEOUT, LIB_TIMEOUT) if timeout_probe else (BUILD, LIB)
    os.makedirs(build_dir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    hdr_t = _deps_mtime()
    todo = []
    objs = []
    for s in srcs:
        obj = os.path.join(build_dir, os.path.basename(s)[:-3] + ".o")
        objs.append(obj)
        if force or verbose_ptxas or not os.path.exists(obj) or \
                os.path.getmtime(obj) < max(os.path.getmtime(s), hdr_t):
            todo.append((s, obj))

    def compile_one(item):
        s, obj = item
        tmp = obj + f".tmp{os.getpid()}"
        cmd = [nvcc(), "-c", s, "-o", tmp] + _flags(verbose_ptxas, bounds_check, timeout_probe)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(s)}:\n{r.stderr}")
        os.replace(tmp, obj)
        return r.stderr

    if todo:
        with cf.ThreadPoolExecutor(max_workers=jobs or min(len(todo), os.cpu_count() or 4)) as ex:
            for err in ex.map(compile_one, todo):
                if verbose_ptxas and err:
                    sys.stderr.write(err)
    if todo or force or not os.path.exists(lib_path) or \
            os.path.getmtime(lib_path) < max(os.path.getmtime(o) for o in objs):
        tmp = lib_path + f".tmp{os.getpid()}"
        cmd = [nvcc(), "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "shared"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv,
                bounds_check="--bounds" in sys.argv))
