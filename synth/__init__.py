"""Seeded, counter-based synthetic inputs (definition in synth.h).

Shared by the tests, the benchmark and the CPU oracle's streaming checks; it
holds none of the optimizer step's arithmetic.  Host fills run in plain C
(libsynth_host.so); device fills (libsynth_cuda.so) write the same bits
straight into GPU memory, so full-size workloads never pass through host RAM.
"""

import ctypes
import math
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
HOST_LIB = os.path.join(HERE, "libsynth_host.so")
CUDA_LIB = os.path.join(HERE, "libsynth_cuda.so")

# output encodings (synth_kinds.h)
OUT_F32, OUT_BF16, OUT_F16, OUT_F32_OF_BF16, OUT_F32_OF_F16 = 0, 1, 2, 3, 4
# stream ids (synth.h)
STREAM_GRAD, STREAM_PARAM, STREAM_EXP_AVG, STREAM_EXP_AVG_SQ, STREAM_AUX = 1, 2, 3, 4, 5

_host = None
_cuda = None


def _fresh(lib, deps):
    return os.path.exists(lib) and all(os.path.getmtime(lib) >= os.path.getmtime(d) for d in deps)


def build_host(force=False):
    src = os.path.join(HERE, "synth_host.c")
    deps = [src, os.path.join(HERE, "synth.h"), os.path.join(HERE, "synth_kinds.h")]
    if force or not _fresh(HOST_LIB, deps):
        subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                        src, "-o", HOST_LIB + ".tmp"], check=True)
        os.replace(HOST_LIB + ".tmp", HOST_LIB)
    return HOST_LIB


def build_cuda(force=False):
    src = os.path.join(HERE, "synth_cuda.cu")
    deps = [src, os.path.join(HERE, "synth.h"), os.path.join(HERE, "synth_kinds.h")]
    if force or not _fresh(CUDA_LIB, deps):
        subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
                        "-lineinfo", "-Xcompiler", "-fPIC", "-shared", src,
                        "-o", CUDA_LIB + ".tmp"], check=True)
        os.replace(CUDA_LIB + ".tmp", CUDA_LIB)
    return CUDA_LIB


def host():
    global _host
    if _host is None:
        L = ctypes.CDLL(build_host())
        U64, U32, I32, I64, F, P = (ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int32,
                                    ctypes.c_int64, ctypes.c_float, ctypes.c_void_p)
        L.synth_key_for.argtypes = [U64, U32, U32, U32]
        L.synth_key_for.restype = U64
        L.synth_fill_normal.argtypes = [P, I32, I64, U64, U64, F]
        L.synth_fill_normal.restype = None
        L.synth_fill_uniform_f32.argtypes = [P, I64, U64, U64, F]
        L.synth_fill_uniform_f32.restype = None
        L.synth_bits_at.argtypes = [U64, U64]
        L.synth_bits_at.restype = U64
        L.synth_gather_normal.argtypes = [P, I32, P, I64, U64, F]
        L.synth_gather_normal.restype = None
        _host = L
    return _host


def cuda():
    """The device-fill library; raises if it was not built."""
    global _cuda
    if _cuda is None:
        if not os.path.exists(CUDA_LIB):
            raise RuntimeError(f"{CUDA_LIB} missing: run __graft_entry__.build()")
        L = ctypes.CDLL(CUDA_LIB)
        U64, I32, I64, F, P = (ctypes.c_uint64, ctypes.c_int32, ctypes.c_int64,
                               ctypes.c_float, ctypes.c_void_p)
        L.synth_cuda_fill_normal.argtypes = [P, I32, I64, U64, U64, F, P]
        L.synth_cuda_fill_normal.restype = ctypes.c_int
        L.synth_cuda_fill_uniform_f32.argtypes = [P, I64, U64, U64, F, P]
        L.synth_cuda_fill_uniform_f32.restype = ctypes.c_int
        _cuda = L
    return _cuda


def factor(sigma):
    """fp32 factor turning the centred Irwin-Hall integer into N(0, sigma^2) scale."""
    return float(np.float32(sigma / math.sqrt((2.0**32 - 1.0) / 3.0)))


def key(seed, stream, step, replica):
    return int(host().synth_key_for(seed, stream, step, replica))


def normal(n, key_, index0=0, sigma=1.0, kind=OUT_F32):
    """n values of the generator stream `key_`, from index index0."""
    dt = np.uint16 if kind in (OUT_BF16, OUT_F16) else np.float32
    out = np.empty(n, dtype=dt)
    if n:
        host().synth_fill_normal(out.ctypes.data, kind, n, key_, index0, factor(sigma))
    return out


def normal_at(indices, key_, sigma=1.0, kind=OUT_F32):
    """Values of stream `key_` at the given element indices."""
    idx = np.ascontiguousarray(indices, dtype=np.uint64)
    dt = np.uint16 if kind in (OUT_BF16, OUT_F16) else np.float32
    out = np.empty(len(idx), dtype=dt)
    if len(idx):
        host().synth_gather_normal(out.ctypes.data, kind, idx.ctypes.data, len(idx), key_,
                                   factor(sigma))
    return out


def uniform(n, key_, index0=0, scale=1.0):
    out = np.empty(n, dtype=np.float32)
    if n:
        host().synth_fill_uniform_f32(out.ctypes.data, n, key_, index0, scale)
    return out


def cuda_normal_(dev_ptr, n, key_, index0=0, sigma=1.0, kind=OUT_F32, stream=0):
    """Fills n device elements at dev_ptr; stream is a cudaStream_t as int."""
    rc = cuda().synth_cuda_fill_normal(ctypes.c_void_p(dev_ptr), kind, n, key_, index0,
                                       factor(sigma), ctypes.c_void_p(stream))
    if rc != 0:
        raise RuntimeError(f"synth_cuda_fill_normal failed: cudaError {rc}")


def cuda_uniform_(dev_ptr, n, key_, index0=0, scale=1.0, stream=0):
    rc = cuda().synth_cuda_fill_uniform_f32(ctypes.c_void_p(dev_ptr), n, key_, index0,
                                            scale, ctypes.c_void_p(stream))
    if rc != 0:
        raise RuntimeError(f"synth_cuda_fill_uniform_f32 failed: cudaError {rc}")
