"""Builds libvpp.so (sm_103a) in-tree: one nvcc -c per .cu file, in parallel,
then one shared-library link with the CUDA runtime linked statically."""

from __future__ import annotations

import concurrent.futures
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libvpp.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
         "-I" + INCLUDE, "-I" + CSRC]


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale(obj, src, hdr_mtime):
    return (not os.path.exists(obj) or os.path.getmtime(obj) < os.path.getmtime(src)
            or os.path.getmtime(obj) < hdr_mtime)


def build(verbose: bool = False, jobs: int | None = None, extra_flags=(), out_dir: str | None = None,
          lib_name: str = "libvpp.so") -> str:
    """Compiles what changed and (re)links the library; returns its path.

    The default is the product library, _build/libvpp.so.  A different
    out_dir with extra_flags builds a variant beside it (for example a
    tracing build) without touching the product's objects."""
    out = out_dir or OUT_DIR
    lib = os.path.join(out, lib_name)
    os.makedirs(out, exist_ok=True)
    nvcc = _nvcc()
    hdr_mtime = max((os.path.getmtime(h) for h in _headers()), default=0.0)
    srcs = _sources()
    objs = [os.path.join(out, os.path.basename(s)[:-3] + ".o") for s in srcs]
    todo = [(s, o) for s, o in zip(srcs, objs) if _stale(o, s, hdr_mtime)]

    def compile_one(so):
        s, o = so
        cmd = [nvcc, *ARCH, *FLAGS, *extra_flags, "-c", s, "-o", o]
        if verbose:
            cmd.append("-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(s)}:\n{r.stdout}\n{r.stderr}")
        return s, r.stderr

    if todo:
        n = jobs or min(len(todo), os.cpu_count() or 4)
        with concurrent.futures.ThreadPoolExecutor(max_workers=n) as ex:
            for s, err in ex.map(compile_one, todo):
                if verbose and err:
                    sys.stderr.write(f"--- {os.path.basename(s)}\n{err}")
    if todo or not os.path.exists(lib) or any(os.path.getmtime(lib) < os.path.getmtime(o) for o in objs):
        tmp = lib + ".tmp"
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs, "-ldl", "-lpthread", "-lrt"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
