"""CPU oracle of the sharded mixed-precision Adam step.  TEST INFRASTRUCTURE ONLY.

Only tests/, the smoke check (__graft_entry__.smoke) and the CPU-baseline leg
of bench.py may import this package.  The product path (the CUDA library and
its Python binding) never imports it, and it imports nothing of the product.

Parts:
  shard_map.py -- step A1 (buffers, buckets, per-rank views), plain Python.
  oracle.c     -- steps A2..A6 (replica reduction, unscale and inf check,
                  fp64 sum of squares, clip coefficient, AdamW, write-back)
                  and the pre-reduction grad check (largest |g| per replica
                  and bucket), scalar C compiled with -ffp-contract=off.
  step()       -- one optimizer step composed from those parts, in the
                  order of the MixedPrecisionOptimizer step skeleton of the
                  distrib_optimizer page: prepare_grads (copy to fp32 main
                  grad, unscale, inf/NaN) -> skip on inf -> clip_grad_norm ->
                  inner AdamW step -> copy main params back to the model
                  param buffer.
  loss_scale.py -- step A7, the fp16 dynamic loss scale (start at 2^16 from
                  the DeepSpeed setting initial_scale_power 16; backoff on
                  an overflow after the hysteresis strikes, growth after a
                  run of clean steps), plain Python.  With a hysteresis of 1
                  it is pinned to torch's GradScaler update routine and to
                  hand-worked sequences; above 1 only hand-worked sequences
                  pin it.
"""

import ctypes

import numpy as np

from . import build as _build
from .loss_scale import LossScale, initial_scale  # noqa: F401
from .shard_map import BF16, F16, F32, Range, ShardMap, pad_up  # noqa: F401

_lib = None


class Hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double),
                ("beta2", ctypes.c_double), ("eps", ctypes.c_double),
                ("weight_decay", ctypes.c_double)]


def lib():
    """Loads liboracle.so, building it first if needed."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P, I32, I64, F, D = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                             ctypes.c_float, ctypes.c_double)
        L.or_reduce_prepare_run.argtypes = [ctypes.POINTER(P), I32, I32, I32, I32, I64, I64, F, F, P]
        L.or_reduce_prepare_run.restype = I64
        L.or_grad_amax_run.argtypes = [P, I32, I64, I64]
        L.or_grad_amax_run.restype = D
        L.or_sumsq_run.argtypes = [P, I64]
        L.or_sumsq_run.restype = D
        L.or_clip_coef.argtypes = [D, D, ctypes.POINTER(D), ctypes.POINTER(D)]
        L.or_clip_coef.restype = I32
        L.or_adamw_run.argtypes = [P, I64, D, I32, P, P, P, ctypes.POINTER(Hparams), D, I64, P, I32]
        L.or_adamw_run.restype = None
        L.or_stream_sumsq.argtypes = [ctypes.POINTER(ctypes.c_uint64), I32, I32, I32, I32, F,
                                      ctypes.c_uint64, I64, F, F, ctypes.POINTER(I64)]
        L.or_stream_sumsq.restype = D
        L.or_stream_reduce_prepare_run.argtypes = [ctypes.POINTER(ctypes.c_uint64), I32, I32, I32, I32, F,
                                                   ctypes.c_uint64, I64, F, F, P]
        L.or_stream_reduce_prepare_run.restype = I64
        L.or_round_bf16.argtypes = [F]
        L.or_round_bf16.restype = ctypes.c_uint16
        L.or_round_f16.argtypes = [F]
        L.or_round_f16.restype = ctypes.c_uint16
        L.or_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.or_bf16_to_f32.restype = F
        L.or_f16_to_f32.argtypes = [ctypes.c_uint16]
        L.or_f16_to_f32.restype = F
        _lib = L
    return _lib


def ctypes_byref(x):
    return ctypes.byref(x)


def ctypes_double(v=0.0):
    return ctypes.c_double(v)


def _ptr(a, offset=0):
    return ctypes.c_void_p(a.ctypes.data + offset * a.itemsize)


def _f32_args(x):
    # each value handed over as its fp32 bit pattern: a trip through a Python
    # float (a double) would quiet a signalling NaN before the cast sees it
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32).ravel())
    return [ctypes.c_float.from_buffer_copy(x[i:i + 1].tobytes()) for i in range(x.size)]


def round_bf16(x):
    """RNE fp32 -> bfloat16 bits, elementwise (oracle's own definition)."""
    L = lib()
    return np.array([L.or_round_bf16(v) for v in _f32_args(x)], dtype=np.uint16)


def round_f16(x):
    """RNE fp32 -> binary16 bits, elementwise (oracle's own definition)."""
    L = lib()
    return np.array([L.or_round_f16(v) for v in _f32_args(x)], dtype=np.uint16)


def reduce_prepare(replicas, gdt, index0, length, inv_scale, n_inst=1, average=False,
                   grad_scale=1.0):
    """A2 (+ A2' scale_gradients) + A3 on a run: returns (main grads fp32,
    count of non-finite)."""
    L = lib()
    n = len(replicas)
    arr = (ctypes.c_void_p * n)(*[r.ctypes.data for r in replicas])
    out = np.empty(length, dtype=np.float32)
    bad = L.or_reduce_prepare_run(arr, n, n_inst, gdt, int(average), index0, length,
                                  grad_scale, inv_scale, _ptr(out))
    if bad < 0:
        raise ValueError("invalid replica / instance counts")
    return out, bad


def grad_amax_run(rep, gdt, index0, length):
    """The pre-reduction grad check over a run of one replica (see
    or_grad_amax_run): NaN if the run holds a NaN, else the largest |g|."""
    return lib().or_grad_amax_run(_ptr(rep), gdt, index0, length)


def bucket_number(smap, bi, b):
    """Number of bucket b of buffer bi among all buffers' buckets."""
    return sum(len(buf.buckets) for buf in smap.buffers[:bi]) + b


def _amax_merge(a, b):
    return float("nan") if (a != a or b != b) else max(a, b)


def step(smap, ranks, grads, state, params, hp, t, *, inv_scale=1.0, max_norm=1.0,
         layout="full", n_inst=1, average=False, remote_sumsq=0.0,
         remote_found_inf=False, grad_scale=1.0, check_grads=False):
    """One optimizer step over the shards of `ranks` in every buffer of `smap`.

    grads[bi]  : list of n_rep replica arrays for buffer bi, in its grad dtype
                 (fp32 as float32, bf16/fp16 as uint16 bits).  layout "full":
                 each is the whole grad buffer (numel); layout "shard": each
                 is the flat shard of the single rank in `ranks`.
    state[bi]  : dict with "exp_avg", "exp_avg_sq" and, for a bf16/fp16
                 buffer, "master": float32 arrays of len(ranks) * shard_numel,
                 rank-major (the slot of ranks[i] starts at i * shard_numel).
    params[bi] : the param buffer (numel) in the param dtype; for an fp32
                 buffer it is also the master (updated in place).
    hp         : dict lr, beta1, beta2, eps, weight_decay.
    t          : the step number used for bias correction if not skipped.
    grad_scale : scale_gradients factor applied to the reduced grads (1 = none).
    check_grads: also return grad_amax, the pre-reduction check of every
                 replica: an (n_rep, total buckets) float64 array holding, per
                 replica and bucket, the largest |g| among the elements the
                 step reads (NaN if one is NaN; 0 when it reads none).
    Arrays in state and params are updated in place.  Returns a dict with
    found_inf, norm (NaN when skipped), coef, clip, main (per buffer),
    sumsq and num_zeros (main grads equal to zero, Megatron's count_zeros).
    """
    L = lib()
    n_rep = len(grads[0]) if grads else 0
    mains = []
    sumsq = 0.0
    bad = 0
    zeros = 0
    pieces = []
    amax = np.zeros((n_rep, bucket_number(smap, len(smap.buffers), 0)))
    for bi, buf in enumerate(smap.buffers):
        S = smap.shard_numel(bi)
        main = np.zeros(len(ranks) * S, dtype=np.float32)
        reps = grads[bi]
        arr = (ctypes.c_void_p * n_rep)(*[r.ctypes.data for r in reps])
        for slot, r in enumerate(ranks):
            for pid, b, v in smap.rank_pieces(bi, r):
                n = v["gbuf_local"].size
                local = slot * S + v["shard_offset"]
                rep0 = v["gbuf_world"].start if layout == "full" else v["shard_offset"]
                k = L.or_reduce_prepare_run(arr, n_rep, n_inst, buf.grad_dtype, int(average),
                                            rep0, n, ctypes.c_float(grad_scale),
                                            ctypes.c_float(inv_scale), _ptr(main, local))
                if k < 0:
                    raise ValueError("invalid replica / instance counts")
                bad += k
                if check_grads:
                    col = bucket_number(smap, bi, b)
                    for q in range(n_rep):
                        amax[q, col] = _amax_merge(amax[q, col],
                                                   L.or_grad_amax_run(_ptr(reps[q]), buf.grad_dtype, rep0, n))
                sumsq += L.or_sumsq_run(_ptr(main, local), n)
                zeros += int(np.count_nonzero(main[local:local + n] == 0))
                pieces.append((bi, pid, local, v))
        mains.append(main)
    sumsq += remote_sumsq
    found = bad > 0 or bool(remote_found_inf)
    result = {"found_inf": found, "main": mains, "sumsq": sumsq, "num_zeros": zeros}
    if check_grads:
        result["grad_amax"] = amax
    if found:
        result.update(norm=float("nan"), coef=1.0, clip=False)
        return result
    norm = ctypes.c_double()
    coef = ctypes.c_double()
    clip = L.or_clip_coef(sumsq, max_norm, ctypes.byref(norm), ctypes.byref(coef))
    h = Hparams(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"])
    for bi, pid, local, v in pieces:
        buf = smap.buffers[bi]
        st = state[bi]
        n = v["gbuf_local"].size
        wd_mult = float(smap.params[pid].get("wd_mult", 1.0))
        world = v["gbuf_world"].start
        if buf.param_dtype == F32:
            master_ptr = _ptr(params[bi], world)
            out_ptr = None
        else:
            master_ptr = _ptr(st["master"], local)
            out_ptr = _ptr(params[bi], world)
        L.or_adamw_run(_ptr(mains[bi], local), n, coef.value, clip, master_ptr,
                       _ptr(st["exp_avg"], local), _ptr(st["exp_avg_sq"], local),
                       ctypes.byref(h), wd_mult, t, out_ptr, buf.param_dtype)
    result.update(norm=norm.value, coef=coef.value, clip=bool(clip))
    return result


def stream_sumsq(keys, gdt, factor, index0, length, inv_scale=1.0, n_inst=1, average=False,
                 grad_scale=1.0):
    """A2 + A3 + the fp64 sum of squares over a run whose replica gradients
    are drawn from the seeded generator (keys: one generator key per replica).
    Returns (sumsq, count of non-finite main grads)."""
    L = lib()
    n = len(keys)
    karr = (ctypes.c_uint64 * n)(*keys)
    bad = ctypes.c_int64()
    s = L.or_stream_sumsq(karr, n, n_inst, gdt, int(average), ctypes.c_float(factor),
                          index0, length, ctypes.c_float(grad_scale), ctypes.c_float(inv_scale),
                          ctypes.byref(bad))
    if bad.value < 0:
        raise ValueError("invalid replica / instance counts")
    return s, bad.value


def stream_reduce_prepare(keys, gdt, factor, index0, length, out=None, inv_scale=1.0, n_inst=1,
                          average=False, grad_scale=1.0):
    """A2 + A3 over a run whose replica gradients are drawn from the seeded
    generator (keys: one generator key per replica), keeping the main grads.
    Writes them to `out` (a float32 array of `length`, allocated when None)
    and returns (out, count of non-finite main grads)."""
    L = lib()
    n = len(keys)
    karr = (ctypes.c_uint64 * n)(*keys)
    if out is None:
        out = np.empty(length, dtype=np.float32)
    assert out.dtype == np.float32 and out.flags.c_contiguous and out.size >= length
    bad = L.or_stream_reduce_prepare_run(karr, n, n_inst, gdt, int(average), ctypes.c_float(factor),
                                         index0, length, ctypes.c_float(grad_scale),
                                         ctypes.c_float(inv_scale), _ptr(out))
    if bad < 0:
        raise ValueError("invalid replica / instance counts")
    return out, bad


def float_ulp_diff(a, b):
    """Distance in units of last place between float32 arrays (same sign)."""
    ai = np.asarray(a, dtype=np.float32).view(np.int32).astype(np.int64)
    bi = np.asarray(b, dtype=np.float32).view(np.int32).astype(np.int64)
    ai = np.where(ai < 0, -(ai & 0x7FFFFFFF), ai)
    bi = np.where(bi < 0, -(bi & 0x7FFFFFFF), bi)
    return np.abs(ai - bi)


def master_close(got, want, before, scale_floor, ulps=4):
    """Tolerance test for updated fp32 master weights: |got - want| within
    `ulps` units in the last place of the operand scale max(|before|, |want|,
    scale_floor).  The update p*decay - step*m/denom can cancel, leaving a
    result far smaller than its operands; a few ulps of the operands is then
    the error one rounding difference upstream can cause."""
    got = np.asarray(got, np.float32)
    want = np.asarray(want, np.float32)
    scale = np.maximum(np.maximum(np.abs(before), np.abs(want)), np.float32(scale_floor))
    tol = ulps * np.spacing(scale.astype(np.float32)).astype(np.float64)
    return np.abs(got.astype(np.float64) - want.astype(np.float64)) <= tol


__all__ = ["ShardMap", "Range", "pad_up", "F32", "BF16", "F16", "step", "lib", "LossScale",
           "initial_scale",
           "reduce_prepare", "stream_sumsq", "stream_reduce_prepare", "round_bf16", "round_f16",
           "float_ulp_diff", "master_close"]
