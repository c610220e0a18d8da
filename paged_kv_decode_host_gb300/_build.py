"""Build libpkd.so in-tree with nvcc for sm_103a.

Each translation unit compiles in its own nvcc process (in parallel); the
objects are linked into ``paged_kv_decode_host_gb300/libpkd.so``.  No CMake.
Beside it, when the Python headers are installed, the host C compiler builds
``_pkd_plan``: the binding's argument-marshalling fast path for the per-step
plan calls (the binding falls back to ctypes without it).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
import sysconfig
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpkd.so")
SOURCES = ["planner.cpp", "api.cu", "decode_kernel.cu", "prefix_tc_kernel.cu",
           "merge_kernels.cu", "static_scratch.cu", "append_kernel.cu", "selftest.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
PYPLAN = os.path.join(HERE, "_pkd_plan" + (sysconfig.get_config_var("EXT_SUFFIX") or ".so"))


def _python_include():
    inc = sysconfig.get_paths().get("include")
    return inc if inc and os.path.exists(os.path.join(inc, "Python.h")) else None


def _build_fast_plan():
    """The CPython plan fast path; None when no Python headers or C compiler."""
    inc = _python_include()
    cc = shutil.which("cc") or shutil.which("gcc")
    if inc is None or cc is None:
        return None
    tmp = PYPLAN + f".tmp{os.getpid()}"
    r = subprocess.run([cc, "-O2", "-shared", "-fPIC", f"-I{inc}",
                        os.path.join(CSRC, "pyplan.c"), "-o", tmp], capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(f"_pkd_plan not built (ctypes path used):\n{r.stderr}\n")
        return None
    os.replace(tmp, PYPLAN)
    return PYPLAN


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags():
    return ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
            "-Xcompiler", "-fno-strict-aliasing", f"-I{INCLUDE}", f"-I{CSRC}"] + ARCH


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    if _python_include() is not None and not os.path.exists(PYPLAN):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "pkd.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD, src + ".o")
        lang = ["-x", "cu"] if src.endswith(".cu") else []
        cmd = [nvcc, "-c", *lang, os.path.join(CSRC, src), "-o", obj, *_flags(), *extra_flags]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES) + 1) as ex:
        fast = ex.submit(_build_fast_plan)
        objs = list(ex.map(compile_one, SOURCES))
        fast.result()
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, "-shared", "-o", tmp, *objs, *ARCH, "-Xcompiler", "-fPIC", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True,
                extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else ()))
