"""Build ``libkda.so`` (the CUDA library) and its debug variant
``libkda_debug.so`` in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` file is compiled to an object in parallel, then the
objects are linked into one shared library next to this file.  The debug
variant recompiles the files that hold KDA_DEBUG code with ``-DKDA_DEBUG``
(input precondition and device index checks, see include/kda.h) and shares
the other objects.  The CUDA runtime is linked statically, so the libraries
need only the driver at run time.  Run
``python -m kimi_delta_attention_chunked_gb300.build``.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(PKG, "libkda.so")
LIB_DEBUG_PATH = os.path.join(PKG, "libkda_debug.so")
DEBUG_SOURCES = ("kda_api.cu", "prefill_tc.cu")      # the files with KDA_DEBUG code
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the KDA CUDA library cannot be built")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _fingerprint() -> str:
    h = hashlib.sha256()
    for f in _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + [os.path.join(INCLUDE, "kda.h")]:
        h.update(f.encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(ARCH + NVCC_FLAGS).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile every .cu file under csrc/ and link libkda.so and libkda_debug.so;
    returns libkda.so's path."""
    fp = _fingerprint()
    stamp = LIB_PATH + ".sha256"
    if (not force and all(os.path.exists(p) for p in (LIB_PATH, LIB_DEBUG_PATH, stamp))
            and open(stamp).read() == fp):
        return LIB_PATH
    os.makedirs(os.path.join(BUILD_DIR, "debug"), exist_ok=True)
    cc = nvcc()

    def compile_one(job):
        src, debug = job
        sub = "debug" if debug else ""
        obj = os.path.join(BUILD_DIR, sub, os.path.basename(src) + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra_flags, *(["-DKDA_DEBUG"] if debug else []), "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, flush=True)
        return obj

    srcs = _sources()
    # the two slowest files first, so that they start at once
    jobs = sorted([(f, False) for f in srcs] + [(f, True) for f in srcs if os.path.basename(f) in DEBUG_SOURCES],
                  key=lambda j: os.path.basename(j[0]) != "prefill_tc.cu")
    with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        objs = dict(zip(jobs, ex.map(compile_one, jobs)))

    def link(path, debug):
        members = [objs[(f, debug and os.path.basename(f) in DEBUG_SOURCES)] for f in srcs]
        tmp = path + f".tmp{os.getpid()}"
        r = subprocess.run([cc, *ARCH, "-shared", "-cudart", "static", *members, "-o", tmp], capture_output=True,
                           text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of {os.path.basename(path)} failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, path)

    link(LIB_PATH, False)
    link(LIB_DEBUG_PATH, True)
    with open(stamp, "w") as fh:
        fh.write(fp)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
