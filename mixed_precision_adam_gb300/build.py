"""Builds the in-tree CUDA library lib/libdopt.so for sm_103a.

Six translation units (the host shard map in C++; the device entry points
and the finalize kernel; the reduce/prepare kernels for each of the three
grad dtypes; the AdamW kernel) are compiled in parallel and linked into one
shared library with the CUDA runtime linked statically.  Run this file as a script
(python mixed_precision_adam_gb300/build.py) or call build().
"""

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIBDIR = os.path.join(HERE, "lib")
LIB = os.path.join(LIBDIR, "libdopt.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE]
SOURCES = ["shard_map.cpp", "dopt_cuda.cu", "k1_f32.cu", "k1_bf16.cu", "k1_f16.cu", "k3.cu"]


def _deps():
    out = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    out.append(os.path.join(INCLUDE, "dopt.h"))
    return out


def build(force=False, verbose=False, extra_flags=()):
    if not force and os.path.exists(LIB) and all(
            os.path.getmtime(LIB) >= os.path.getmtime(d) for d in _deps()):
        return LIB
    os.makedirs(LIBDIR, exist_ok=True)
    objs, procs = [], []
    for src in SOURCES:
        obj = os.path.join(LIBDIR, src + ".o")
        cmd = ["nvcc", *ARCH, *NVCC_FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if src.endswith(".cu") and verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        objs.append(obj)
    for cmd, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode:
            sys.stdout.write(out.decode())
        if p.returncode:
            raise RuntimeError("compile failed: " + " ".join(cmd))
    tmp = LIB + ".tmp"
    subprocess.run(["nvcc", *ARCH, "-shared", *objs, "-o", tmp], check=True)
    os.replace(tmp, LIB)
    for o in objs:
        os.remove(o)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose="-v" in sys.argv))
