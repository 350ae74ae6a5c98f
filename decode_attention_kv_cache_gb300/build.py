"""Build libkvc.so in-tree: every .cu under csrc/ compiled for sm_103a in parallel, then linked.

    python -m decode_attention_kv_cache_gb300.build

Objects go to _build/ next to this file; the library to libkvc.so next to this
file.  The CUDA runtime is linked statically, and the driver's tensor-map
encoder is fetched at run time, so the library needs no -lcuda.  No fast-math:
the quantiser depends on IEEE division.

build(trace=True) makes the diagnostic variant libkvc_trace.so (objects in
_build_trace/), compiled with -DKVC_TRACE: the decode split pass then records
clock stamps of its pipeline events (see trace_kernels.py).  The product build
never defines it.
"""

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libkvc.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", os.path.join(HERE, "..", "include")]


def nvcc():
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkvc")
    return exe


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _compile(src, build_dir=BUILD, extra=()):
    obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc()] + ARCH + FLAGS + list(extra) + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, r.stdout, r.stderr))
    return obj


def build(verbose=False, trace=False):
    build_dir = BUILD + ("_trace" if trace else "")
    lib = os.path.join(HERE, "libkvc_trace.so") if trace else LIB
    extra = ("-DKVC_TRACE",) if trace else ()
    os.makedirs(build_dir, exist_ok=True)
    srcs = sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(lambda src: _compile(src, build_dir, extra), srcs))
    tmp = lib + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib)
    if verbose:
        print("built", lib)
    return lib


if __name__ == "__main__":
    build(verbose=True)
    sys.exit(0)
