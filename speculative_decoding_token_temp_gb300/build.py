"""Build step of the CUDA library: one nvcc invocation, sm_103a only, in-tree output.

The library is plain C ABI (include/spec_verify.h) with the CUDA runtime linked
statically, so the Python layer loads it with ctypes and nothing else."""
from __future__ import annotations

import hashlib
import os
import platform
import shutil
import subprocess
import sys
import time

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


def _nvcc_version() -> str:
    try:
        out = subprocess.run([nvcc_path(), "--version"], capture_output=True, text=True, timeout=60).stdout
    except (OSError, subprocess.SubprocessError):
        return "unknown"
    return out.strip().splitlines()[-1] if out.strip() else "unknown"


def build_key(lib: str = LIB) -> str:
    """What a library build depends on: the bytes of every input, the command line, the
    machine architecture (a library built on another host does not load here) and the
    compiler's version."""
    h = hashlib.sha256()
    for f in _inputs():
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(_command(lib, False)[1:]).encode())
    h.update(platform.machine().encode())
    h.update(_nvcc_version().encode())
    return h.hexdigest()


def _stamp(lib: str) -> str:
    return lib + ".stamp"


def up_to_date(lib: str = LIB) -> bool:
    """The library exists and its stamp records the current build key."""
    if not os.path.exists(lib) or not os.path.exists(_stamp(lib)):
        return False
    with open(_stamp(lib)) as f:
        return f.read().split()[0:1] == [build_key(lib)]


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
    t0 = time.time()
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
        with open(_stamp(lib), "w") as f:
            f.write(f"{build_key(lib)} {platform.machine()} sm_103a\n")
    if failed:
        raise RuntimeError("\n".join(failed))
    names = ", ".join(os.path.basename(x) for x in todo)
    print(f"[build] {'compiled ' + names + f' for sm_103a on {platform.machine()} in {time.time() - t0:.0f} s' if todo else 'libraries up to date'}",
          file=sys.stderr)
    return LIB


if __name__ == "__main__":
    import sys
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas-info" in sys.argv,
          bounds="--no-bounds" not in sys.argv)
