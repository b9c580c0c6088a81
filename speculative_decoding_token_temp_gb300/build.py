"""Build step of the CUDA library: one nvcc invocation, sm_103a only, in-tree output.

The library is plain C ABI (include/spec_verify.h) with the CUDA runtime linked
statically, so the Python layer loads it with ctypes and nothing else."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
INCLUDE = os.path.join(ROOT, "include")
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libspecverify.so")
# the same library with every computed access bounds-checked (SPEC_BOUNDS_CHECK=1): a debug
# variant for tests, which reports an access outside its buffer as SPEC_DEV_BOUNDS
LIB_BOUNDS = os.path.join(PKG, "libspecverify_bounds.so")
SOURCES = ["spec_verify.cu"]
HEADERS = ["kernels.cuh", "kernels_rows.cuh", "kernels_sample.cuh", "kernels_multi.cuh", "plan.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _inputs():
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "spec_verify.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _command(lib: str, ptxas_info: bool) -> list:
    cmd = [nvcc_path(), *ARCH, "-lineinfo", "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-cudart", "static", "-I", INCLUDE, "-I", CSRC, "-o", lib + ".tmp"]
    if lib == LIB_BOUNDS:
        cmd.append("-DSPEC_BOUNDS_CHECK=1")
    if ptxas_info:
        cmd += ["-Xptxas", "-v"]
    return cmd + [os.path.join(CSRC, s) for s in SOURCES]


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, bounds: bool = True) -> str:
    """Compile csrc/*.cu into libspecverify.so next to this file and, with bounds, the
    bounds-checked variant libspecverify_bounds.so beside it (the two nvcc runs in
    parallel); return the path of the ordinary library."""
    libs = [LIB] + ([LIB_BOUNDS] if bounds else [])
    todo = [lib for lib in libs if force or not up_to_date(lib)]
    procs = []
    for lib in todo:
        cmd = _command(lib, ptxas_info)
        if verbose:
            print(" ".join(cmd))
        procs.append((lib, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)))
    failed = []
    for lib, proc in procs:
        out, err = proc.communicate()
        if proc.returncode != 0:
            failed.append(f"{os.path.basename(lib)}: nvcc failed ({proc.returncode}):\n{out}\n{err}")
            continue
        if verbose or ptxas_info:
            print(out + err)
        os.replace(lib + ".tmp", lib)
    if failed:
        raise RuntimeError("\n".join(failed))
    return LIB


if __name__ == "__main__":
    import sys
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas-info" in sys.argv,
          bounds="--no-bounds" not in sys.argv)
