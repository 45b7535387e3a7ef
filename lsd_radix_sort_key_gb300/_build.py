"""Compile the CUDA library (csrc/*.cu) into _lib/librs.so for sm_103a.

One translation unit per key type plus the C-ABI unit, compiled in parallel
with nvcc, then linked into a shared library with the CUDA runtime linked
statically.  Nothing here runs at import time of the package except the
check that the library exists.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIBDIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIBDIR, "librs.so")
INCLUDE = os.path.join(ROOT, "include")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return path


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
    deps += glob.glob(os.path.join(INCLUDE, "*.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, extra_flags=(), verbose: bool = False, libdir: str | None = None) -> str:
    """Build librs.so if any source is newer than it; returns its path.

    extra_flags / libdir build a variant (e.g. -D switches) into another folder.
    """
    out_dir = libdir or LIBDIR
    out_lib = os.path.join(out_dir, "librs.so")
    if not force and libdir is None and not _stale():
        return LIB
    os.makedirs(out_dir, exist_ok=True)
    objdir = os.path.join(out_dir, "obj")
    os.makedirs(objdir, exist_ok=True)
    common = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-I", INCLUDE, "-I", CSRC, *extra_flags]

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        cmd = common + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = out_lib + f".{os.getpid()}.tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out_lib)
    return out_lib


if __name__ == "__main__":
    # python -m lsd_radix_sort_key_gb300._build [--libdir DIR --flags "-DNAME=VALUE ..."]
    # builds the library, or a variant of it (compile-time switches, e.g. the
    # shapes in rs_config.h) into DIR, and prints the library's path.
    import argparse
    import shlex
    ap = argparse.ArgumentParser()
    ap.add_argument("--libdir", default=None)
    ap.add_argument("--flags", default="")
    a = ap.parse_args()
    print(build(force=True, verbose=True, extra_flags=shlex.split(a.flags), libdir=a.libdir))
