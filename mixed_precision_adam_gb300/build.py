"""Builds the in-tree CUDA library lib/libdopt.so for sm_103a.

Six translation units (the host shard map in C++; the device entry points
and the finalize kernel; the reduce/prepare kernels for each of the three
grad dtypes; the AdamW kernel) are compiled in parallel and linked into one
shared library with the CUDA runtime linked statically.  Run this file as a script
(python mixed_precision_adam_gb300/build.py) or call build().

build_checked() builds the same sources with DOPT_BOUNDS_CHECK=1 into
lib/libdopt_checked.so: a debug build whose kernels check every tile
against the extents of its buffers (dopt_debug_bounds_record), which the
tests load through DOPT_LIBRARY.
"""

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIBDIR = os.path.join(HERE, "lib")
LIB = os.path.join(LIBDIR, "libdopt.so")
CHECKED_LIB = os.path.join(LIBDIR, "libdopt_checked.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE]
SOURCES = ["shard_map.cpp", "dopt_cuda.cu", "k1_f32.cu", "k1_bf16.cu", "k1_f16.cu", "k3.cu"]


def _deps():
    out = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    out.append(os.path.join(INCLUDE, "dopt.h"))
    return out


def build(force=False, verbose=False, extra_flags=(), out=LIB):
    if not force and os.path.exists(out) and all(
            os.path.getmtime(out) >= os.path.getmtime(d) for d in _deps()):
        return out
    os.makedirs(LIBDIR, exist_ok=True)
    tag = os.path.splitext(os.path.basename(out))[0]
    objs, procs = [], []
    for src in SOURCES:
        obj = os.path.join(LIBDIR, f"{tag}.{src}.o")
        cmd = ["nvcc", *ARCH, *NVCC_FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if src.endswith(".cu") and verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        objs.append(obj)
    for cmd, p in procs:
        log, _ = p.communicate()
        if verbose or p.returncode:
            sys.stdout.write(log.decode())
        if p.returncode:
            raise RuntimeError("compile failed: " + " ".join(cmd))
    tmp = out + ".tmp"
    subprocess.run(["nvcc", *ARCH, "-shared", *objs, "-o", tmp], check=True)
    os.replace(tmp, out)
    for o in objs:
        os.remove(o)
    return out


def build_checked(force=False, verbose=False):
    return build(force, verbose, ("-DDOPT_BOUNDS_CHECK=1",), CHECKED_LIB)


if __name__ == "__main__":
    print(build(force=True, verbose="-v" in sys.argv))
