"""Sharded mixed-precision Adam (ZeRO-1 DistributedOptimizer step) for GB300.

A thin ctypes binding of the C ABI in include/dopt.h: every function keeps its
C name and only marshals arguments (device pointers may be given as ints or
as objects with a data_ptr() method, streams as ints or objects with a
cuda_stream attribute).  All the work runs in lib/libdopt.so; importing this
package fails loudly when the library has not been built.
"""

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
# DOPT_LIBRARY may name another in-tree build of the same library (the
# bounds-checked debug build, libdopt_checked.so): only its file name counts,
# and the file must sit in this package's lib/ directory
LIB_PATH = os.path.join(HERE, "lib", os.path.basename(os.environ.get("DOPT_LIBRARY") or "libdopt.so"))

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with "
                      "`python mixed_precision_adam_gb300/build.py` (or __graft_entry__.build())")

_lib = ctypes.CDLL(LIB_PATH)

F32, BF16, F16 = 0, 1, 2
OK, E_INVALID, E_ALIGN, E_SIZE, E_CUDA, E_NOMEM = 0, -1, -2, -3, -4, -5
GROUP_FP32_FROM_FLOAT16, GROUP_FP32 = 0, 1
LAYOUT_FULL_BUFFER, LAYOUT_SHARD_ONLY, LAYOUT_BUCKET = 0, 1, 2
ALL_RANKS = -1
MAX_REPLICAS = 64

_P, _I32, _I64, _F, _D, _SZ = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                               ctypes.c_float, ctypes.c_double, ctypes.c_size_t)


class dopt_range(ctypes.Structure):
    _fields_ = [("start", _I64), ("end", _I64)]


class dopt_param_desc(ctypes.Structure):
    _fields_ = [("numel", _I64), ("dtype", _I32), ("new_bucket", _I32), ("wd_mult", _D)]


class dopt_buffer_info(ctypes.Structure):
    _fields_ = [("param_dtype", _I32), ("grad_dtype", _I32), ("group", _I32),
                ("n_buckets", _I32), ("n_params", _I32), ("reserved", _I32),
                ("numel", _I64), ("numel_unpadded", _I64), ("shard_numel", _I64)]


class dopt_bucket_info(ctypes.Structure):
    _fields_ = [("offset", _I64), ("numel", _I64), ("numel_unpadded", _I64),
                ("shard_numel", _I64), ("shard_base", _I64)]


class dopt_param_shard(ctypes.Structure):
    _fields_ = [("param", _I32), ("buffer", _I32), ("bucket", _I32), ("rank", _I32),
                ("gbuf_world", dopt_range), ("gbuf_world_in_bucket", dopt_range),
                ("gbuf_local", dopt_range), ("param_range", dopt_range),
                ("shard_offset", _I64)]


class dopt_adamw_hparams(ctypes.Structure):
    _fields_ = [("lr", _D), ("beta1", _D), ("beta2", _D), ("eps", _D),
                ("weight_decay", _D), ("step", _I64)]


class dopt_step_args(ctypes.Structure):
    _fields_ = [("map", _P), ("rank", _I32), ("n_instances", _I32), ("layout", _I32),
                ("average_in_collective", _I32),
                ("replica_grads", ctypes.POINTER(ctypes.POINTER(_P))),
                ("main_grad", ctypes.POINTER(_P)), ("master", ctypes.POINTER(_P)),
                ("exp_avg", ctypes.POINTER(_P)), ("exp_avg_sq", ctypes.POINTER(_P)),
                ("param_buffer", ctypes.POINTER(_P)),
                ("inv_loss_scale", _F), ("remote_found_inf", _I32),
                ("max_norm", _D), ("remote_sumsq", _D), ("hp", dopt_adamw_hparams),
                ("workspace", _P), ("workspace_bytes", _SZ), ("stream", _P),
                ("stage_events", ctypes.POINTER(_P)), ("grad_scale", _F), ("reserved", _I32),
                ("d_step", _P), ("d_lr", _P), ("grad_amax", _P),
                ("d_global_sumsq", _P), ("d_global_found_inf", _P)]


class dopt_step_stats(ctypes.Structure):
    _fields_ = [("sumsq", _D), ("grad_norm", _F), ("clip_coef", _F), ("found_inf", _I32),
                ("clipped", _I32), ("num_zeros", _I64), ("kernel_error", _I32), ("reserved", _I32)]


class dopt_loss_scaler(ctypes.Structure):
    _fields_ = [("scale", _D), ("growth_factor", _D), ("backoff_factor", _D), ("min_scale", _D),
                ("growth_interval", _I32), ("hysteresis", _I32),
                ("growth_tracker", _I32), ("hysteresis_tracker", _I32)]


def _proto(name, res, *args):
    fn = getattr(_lib, name)
    fn.restype = res
    fn.argtypes = list(args)
    return fn


_c = {
    "dopt_build_shard_map": _proto("dopt_build_shard_map", ctypes.c_int,
                                   ctypes.POINTER(dopt_param_desc), _I32, _I32, _I64, _I32, _I32,
                                   ctypes.POINTER(_P)),
    "dopt_shard_map_free": _proto("dopt_shard_map_free", None, _P),
    "dopt_num_buffers": _proto("dopt_num_buffers", _I32, _P),
    "dopt_dp_size": _proto("dopt_dp_size", _I32, _P),
    "dopt_total_buckets": _proto("dopt_total_buckets", _I32, _P),
    "dopt_bucket_number": _proto("dopt_bucket_number", _I32, _P, _I32, _I32),
    "dopt_buffer_info_get": _proto("dopt_buffer_info_get", ctypes.c_int, _P, _I32,
                                   ctypes.POINTER(dopt_buffer_info)),
    "dopt_bucket_info_get": _proto("dopt_bucket_info_get", ctypes.c_int, _P, _I32, _I32,
                                   ctypes.POINTER(dopt_bucket_info)),
    "dopt_param_index": _proto("dopt_param_index", ctypes.c_int, _P, _I32, ctypes.POINTER(_I32),
                               ctypes.POINTER(_I64), ctypes.POINTER(_I64), ctypes.POINTER(_I32)),
    "dopt_rank_shards": _proto("dopt_rank_shards", ctypes.c_int, _P, _I32, _I32,
                               ctypes.POINTER(dopt_param_shard), _I32, ctypes.POINTER(_I32)),
    "dopt_workspace_bytes": _proto("dopt_workspace_bytes", _SZ, _P, _I32),
    "dopt_grad_reduce_shard": _proto("dopt_grad_reduce_shard", ctypes.c_int, _P, _I32, _I32,
                                     ctypes.POINTER(_P), _I32, _I32, _I32, _I32, _P, _P, _SZ, _P),
    "dopt_prepare_grads": _proto("dopt_prepare_grads", ctypes.c_int, _P, _I32, _I32, _F, _P, _P,
                                 _SZ, _P),
    "dopt_grad_norm": _proto("dopt_grad_norm", ctypes.c_int, _P, _I32, _P, _SZ, _D, _I32, _D, _P,
                             _P, _P, _P),
    "dopt_adam_step": _proto("dopt_adam_step", ctypes.c_int, _P, _I32, _I32, _P, _P, _P, _P, _P,
                             ctypes.POINTER(dopt_adamw_hparams), _P, _P, _P),
    "dopt_step": _proto("dopt_step", ctypes.c_int, ctypes.POINTER(dopt_step_args),
                        ctypes.POINTER(_I32), ctypes.POINTER(_F)),
    "dopt_step_async": _proto("dopt_step_async", ctypes.c_int, ctypes.POINTER(dopt_step_args),
                              _P, _P),
    "dopt_step_noalloc": _proto("dopt_step_noalloc", ctypes.c_int, ctypes.POINTER(dopt_step_args),
                                ctypes.POINTER(_I32), ctypes.POINTER(_F)),
    "dopt_model_numel": _proto("dopt_model_numel", _I64, _P, _I32),
    "dopt_state_to_model": _proto("dopt_state_to_model", ctypes.c_int, _P, _I32, _I32, _I32, _P, _P, _P),
    "dopt_state_from_model": _proto("dopt_state_from_model", ctypes.c_int, _P, _I32, _I32, _I32, _P, _P, _P),
    "dopt_step_from_host": _proto("dopt_step_from_host", ctypes.c_int, ctypes.POINTER(dopt_step_args),
                                  _P, _P, ctypes.POINTER(_I32), ctypes.POINTER(_F)),
    "dopt_workspace_bytes_bucketed": _proto("dopt_workspace_bytes_bucketed", _SZ, _P, _I32),
    "dopt_step_reduce_buckets": _proto("dopt_step_reduce_buckets", ctypes.c_int,
                                       ctypes.POINTER(dopt_step_args), _I32, _I32, _I32),
    "dopt_step_finalize": _proto("dopt_step_finalize", ctypes.c_int, ctypes.POINTER(dopt_step_args),
                                 _P, _P),
    "dopt_step_update_buckets": _proto("dopt_step_update_buckets", ctypes.c_int,
                                       ctypes.POINTER(dopt_step_args), _I32, _I32, _I32),
    "dopt_memory_ledger": _proto("dopt_memory_ledger", _I64, _I64, _I32, _I32,
                                 ctypes.POINTER(_I64)),
    "dopt_comm_bytes": _proto("dopt_comm_bytes", _I64, _I64, _I32, _I32, _I32),
    "dopt_loss_scaler_init": _proto("dopt_loss_scaler_init", ctypes.c_int,
                                    ctypes.POINTER(dopt_loss_scaler), _D, _D, _D, _I32, _I32, _D),
    "dopt_loss_scaler_update": _proto("dopt_loss_scaler_update", ctypes.c_int,
                                      ctypes.POINTER(dopt_loss_scaler), _I32),
    "dopt_kernel_launches": _proto("dopt_kernel_launches", ctypes.c_uint64),
    "dopt_step_local_stats": _proto("dopt_step_local_stats", ctypes.c_int, ctypes.POINTER(dopt_step_args), _P, _P),
    "dopt_debug_bounds_record": _proto("dopt_debug_bounds_record", ctypes.c_int, ctypes.POINTER(_I64)),
    "dopt_read_step_stats": _proto("dopt_read_step_stats", ctypes.c_int, _P,
                                   ctypes.POINTER(dopt_step_stats), _P),
    "dopt_last_error": _proto("dopt_last_error", ctypes.c_char_p),
}
# the debug build's test hook (absent from the release library)
if hasattr(_lib, "dopt_debug_starve_copy"):
    _c["dopt_debug_starve_copy"] = _proto("dopt_debug_starve_copy", ctypes.c_int, _I32)


class DoptError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{message} (status {status})")
        self.status = status


def dopt_last_error():
    return _c["dopt_last_error"]().decode()


def _check(status):
    if status < 0:
        raise DoptError(status, dopt_last_error())
    return status


def _ptr(x):
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "__array_interface__"):  # numpy array (host memory)
        return x.__array_interface__["data"][0]
    return int(x)


def _stream(s):
    if s is None:
        return None
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    return int(s)


def _ptr_array(xs):
    return (_P * len(xs))(*[_ptr(x) for x in xs])


class ShardMap:
    """Owner of a dopt_shard_map handle (freed on garbage collection)."""

    def __init__(self, handle):
        self.handle = ctypes.c_void_p(handle)

    def __del__(self):
        if getattr(self, "handle", None) and self.handle.value:
            _c["dopt_shard_map_free"](self.handle)
            self.handle = None

    @property
    def _as_parameter_(self):
        return self.handle


def dopt_build_shard_map(params, dp_size, bucket_size=0, grad_reduce_in_fp32=False,
                         pad_for_high_busbw=False):
    """params: list of dicts with numel, dtype and optional new_bucket, wd_mult."""
    arr = (dopt_param_desc * len(params))()
    for i, p in enumerate(params):
        arr[i] = dopt_param_desc(int(p["numel"]), int(p["dtype"]), int(bool(p.get("new_bucket", False))),
                                 float(p.get("wd_mult", 1.0)))
    out = _P()
    _check(_c["dopt_build_shard_map"](arr, len(params), dp_size, int(bucket_size),
                                      int(bool(grad_reduce_in_fp32)), int(bool(pad_for_high_busbw)),
                                      ctypes.byref(out)))
    return ShardMap(out.value)


def dopt_num_buffers(m):
    return _check(_c["dopt_num_buffers"](m))


def dopt_dp_size(m):
    return _check(_c["dopt_dp_size"](m))


def dopt_total_buckets(m):
    return _check(_c["dopt_total_buckets"](m))


def dopt_bucket_number(m, buffer, bucket):
    return _check(_c["dopt_bucket_number"](m, buffer, bucket))


def _struct_dict(s):
    out = {}
    for name, _ in s._fields_:
        v = getattr(s, name)
        out[name] = (v.start, v.end) if isinstance(v, dopt_range) else v
    return out


def dopt_buffer_info_get(m, buffer):
    info = dopt_buffer_info()
    _check(_c["dopt_buffer_info_get"](m, buffer, ctypes.byref(info)))
    return _struct_dict(info)


def dopt_bucket_info_get(m, buffer, bucket):
    info = dopt_bucket_info()
    _check(_c["dopt_bucket_info_get"](m, buffer, bucket, ctypes.byref(info)))
    return _struct_dict(info)


def dopt_param_index(m, param):
    b, s, e, k = _I32(), _I64(), _I64(), _I32()
    _check(_c["dopt_param_index"](m, param, ctypes.byref(b), ctypes.byref(s), ctypes.byref(e),
                                  ctypes.byref(k)))
    return b.value, s.value, e.value, k.value


def dopt_rank_shards(m, buffer, rank):
    n = _I32()
    _check(_c["dopt_rank_shards"](m, buffer, rank, None, 0, ctypes.byref(n)))
    arr = (dopt_param_shard * max(1, n.value))()
    _check(_c["dopt_rank_shards"](m, buffer, rank, arr, n.value, ctypes.byref(n)))
    return [_struct_dict(arr[i]) for i in range(n.value)]


def dopt_workspace_bytes(m, rank):
    v = _c["dopt_workspace_bytes"](m, rank)
    if v == 0:
        raise DoptError(E_INVALID, dopt_last_error())
    return v


def dopt_grad_reduce_shard(m, buffer, rank, replicas, n_instances, layout, average_in_collective,
                           main_grad, workspace, workspace_bytes, stream=None):
    _check(_c["dopt_grad_reduce_shard"](m, buffer, rank, _ptr_array(replicas), len(replicas),
                                        n_instances, layout, int(bool(average_in_collective)),
                                        _ptr(main_grad), _ptr(workspace), workspace_bytes,
                                        _stream(stream)))


def dopt_prepare_grads(m, buffer, rank, inv_loss_scale, main_grad, workspace, workspace_bytes,
                       stream=None):
    _check(_c["dopt_prepare_grads"](m, buffer, rank, inv_loss_scale, _ptr(main_grad),
                                    _ptr(workspace), workspace_bytes, _stream(stream)))


def dopt_grad_norm(m, rank, workspace, workspace_bytes, remote_sumsq, remote_found_inf, max_norm,
                   d_norm, d_clip_coef, d_found_inf, stream=None):
    _check(_c["dopt_grad_norm"](m, rank, _ptr(workspace), workspace_bytes, remote_sumsq,
                                int(bool(remote_found_inf)), max_norm, _ptr(d_norm),
                                _ptr(d_clip_coef), _ptr(d_found_inf), _stream(stream)))


def _hparams(hp, step):
    return dopt_adamw_hparams(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"],
                              int(step))


def dopt_adam_step(m, buffer, rank, main_grad, master, exp_avg, exp_avg_sq, param_buffer, hp,
                   step, d_clip_coef, d_found_inf, stream=None):
    h = _hparams(hp, step)
    _check(_c["dopt_adam_step"](m, buffer, rank, _ptr(main_grad), _ptr(master), _ptr(exp_avg),
                                _ptr(exp_avg_sq), _ptr(param_buffer), ctypes.byref(h),
                                _ptr(d_clip_coef), _ptr(d_found_inf), _stream(stream)))


class StepArgs:
    """Marshalled dopt_step_args (keeps the pointer arrays alive)."""

    def __init__(self, m, rank, replica_grads, main_grad, master, exp_avg, exp_avg_sq,
                 param_buffer, hp, step, workspace, workspace_bytes, *, n_instances=1,
                 layout=LAYOUT_FULL_BUFFER, average_in_collective=False, inv_loss_scale=1.0,
                 max_norm=1.0, remote_sumsq=0.0, remote_found_inf=False, stream=None,
                 grad_scale=1.0):
        self.map = m
        self._reps = [_ptr_array(r) for r in replica_grads]
        self._rep_arr = (ctypes.POINTER(_P) * len(self._reps))(
            *[ctypes.cast(r, ctypes.POINTER(_P)) for r in self._reps])
        self._main = _ptr_array(main_grad)
        self._master = _ptr_array(master)
        self._m = _ptr_array(exp_avg)
        self._v = _ptr_array(exp_avg_sq)
        self._param = _ptr_array(param_buffer)
        self.c = dopt_step_args()
        c = self.c
        c.map = m.handle
        c.rank = rank
        c.n_instances = n_instances
        c.layout = layout
        c.average_in_collective = int(bool(average_in_collective))
        c.replica_grads = ctypes.cast(self._rep_arr, ctypes.POINTER(ctypes.POINTER(_P)))
        c.main_grad = ctypes.cast(self._main, ctypes.POINTER(_P))
        c.master = ctypes.cast(self._master, ctypes.POINTER(_P))
        c.exp_avg = ctypes.cast(self._m, ctypes.POINTER(_P))
        c.exp_avg_sq = ctypes.cast(self._v, ctypes.POINTER(_P))
        c.param_buffer = ctypes.cast(self._param, ctypes.POINTER(_P))
        c.inv_loss_scale = inv_loss_scale
        c.remote_found_inf = int(bool(remote_found_inf))
        c.max_norm = max_norm
        c.remote_sumsq = remote_sumsq
        c.hp = _hparams(hp, step)
        c.workspace = _ptr(workspace)
        c.workspace_bytes = workspace_bytes
        c.stream = _stream(stream)
        c.grad_scale = grad_scale

    def set_stage_events(self, events):
        """events: None, or 4 CUDA events (objects with cuda_event, or ints)."""
        if events is None:
            self._events = None
            self.c.stage_events = None
            return
        self._events = (_P * 4)(*[getattr(e, "cuda_event", e) for e in events])
        self.c.stage_events = ctypes.cast(self._events, ctypes.POINTER(_P))

    def set_stream(self, stream):
        self.c.stream = _stream(stream)

    def set_replicas(self, buffer, replicas):
        """Points buffer `buffer`'s replica grads at other device memory (the
        same count; e.g. the staging buffers of DOPT_LAYOUT_BUCKET)."""
        arr = self._reps[buffer]
        if len(replicas) != len(arr):
            raise ValueError("replica count differs")
        for k, r in enumerate(replicas):
            arr[k] = _ptr(r)

    def set_device_step(self, d_step, d_lr=None):
        """Use a device int64 step counter (and optionally a device double
        learning rate) instead of the host step number."""
        self.c.d_step = _ptr(d_step)
        self.c.d_lr = _ptr(d_lr)

    def set_global_stats(self, d_sumsq, d_found_inf):
        """Global norm terms in device memory for dopt_step_finalize (a
        device float64 scalar and a device int32 scalar, or None, None)."""
        self._global = (d_sumsq, d_found_inf)
        self.c.d_global_sumsq = _ptr(d_sumsq)
        self.c.d_global_found_inf = _ptr(d_found_inf)

    def set_grad_check(self, grad_amax):
        """Turns on the pre-reduction grad check: grad_amax is a device
        float32 array of n_replicas x dopt_total_buckets(map) (or None to
        turn it off)."""
        self._grad_amax = grad_amax
        self.c.grad_amax = _ptr(grad_amax)

    def set_step(self, step, lr=None):
        self.c.hp.step = int(step)
        if lr is not None:
            self.c.hp.lr = lr


def dopt_step(args):
    """Runs one fused step; returns (found_inf: bool, grad_norm: float)."""
    f, n = _I32(), _F()
    _check(_c["dopt_step"](ctypes.byref(args.c), ctypes.byref(f), ctypes.byref(n)))
    return bool(f.value), n.value


NOALLOC_SCRATCH_BYTES = 1 << 20


def dopt_step_noalloc(args):
    """The fused step with the library's static scratch instead of a
    workspace (args' workspace is ignored); returns (found_inf, grad_norm)."""
    f, n = _I32(), _F()
    _check(_c["dopt_step_noalloc"](ctypes.byref(args.c), ctypes.byref(f), ctypes.byref(n)))
    return bool(f.value), n.value


STATE_FLAT_SHARD, STATE_PARAM_BUFFER = 0, 1


def dopt_model_numel(m, buffer):
    return _check(_c["dopt_model_numel"](m, buffer))


def dopt_state_to_model(m, buffer, rank, layout, state, model, stream=None):
    """Copies the pieces rank (or ALL_RANKS) owns of a state tensor into
    model space (buffer params in model order); device or host arrays."""
    _check(_c["dopt_state_to_model"](m, buffer, rank, layout, _ptr(state), _ptr(model), _stream(stream)))


def dopt_state_from_model(m, buffer, rank, layout, model, state, stream=None):
    """The reverse of dopt_state_to_model."""
    _check(_c["dopt_state_from_model"](m, buffer, rank, layout, _ptr(model), _ptr(state), _stream(stream)))


def dopt_step_from_host(args, host_replica_grads, copy_stream=None):
    """One step whose replica grads start in host memory: host_replica_grads
    is a list per buffer of host arrays (pinned torch tensors or numpy
    arrays) laid out like args' device replicas, which the library fills
    bucket by bucket while it reduces; args needs the bucket-staged
    workspace.  Returns (found_inf, grad_norm)."""
    rows = [_ptr_array(reps) for reps in host_replica_grads]
    table = (ctypes.POINTER(_P) * len(rows))(*[ctypes.cast(r, ctypes.POINTER(_P)) for r in rows])
    f, n = _I32(), _F()
    _check(_c["dopt_step_from_host"](ctypes.byref(args.c), ctypes.cast(table, _P), _stream(copy_stream),
                                     ctypes.byref(f), ctypes.byref(n)))
    return bool(f.value), n.value


def dopt_step_async(args, d_found_inf=None, d_norm=None):
    _check(_c["dopt_step_async"](ctypes.byref(args.c), _ptr(d_found_inf), _ptr(d_norm)))


def dopt_workspace_bytes_bucketed(m, rank):
    v = _c["dopt_workspace_bytes_bucketed"](m, rank)
    if v == 0:
        raise DoptError(E_INVALID, dopt_last_error())
    return v


def dopt_step_reduce_buckets(args, buffer, bucket_first, bucket_count=1):
    _check(_c["dopt_step_reduce_buckets"](ctypes.byref(args.c), buffer, bucket_first, bucket_count))


def dopt_step_finalize(args, d_found_inf=None, d_norm=None):
    _check(_c["dopt_step_finalize"](ctypes.byref(args.c), _ptr(d_found_inf), _ptr(d_norm)))


def dopt_step_local_stats(args, d_local_sumsq, d_local_found_inf):
    """This rank's local sum of squares (device float64) and non-finite flag
    (device int32) after its bucket-staged reduces, for a device all-reduce."""
    _check(_c["dopt_step_local_stats"](ctypes.byref(args.c), _ptr(d_local_sumsq), _ptr(d_local_found_inf)))


def dopt_step_update_buckets(args, buffer, bucket_first, bucket_count=1):
    _check(_c["dopt_step_update_buckets"](ctypes.byref(args.c), buffer, bucket_first, bucket_count))


def dopt_read_step_stats(workspace, stream=None):
    """The last step's statistics (waits for the stream) as a dict."""
    st = dopt_step_stats()
    _check(_c["dopt_read_step_stats"](_ptr(workspace), ctypes.byref(st), _stream(stream)))
    return _struct_dict(st)


def dopt_debug_starve_copy(tile):
    """The bounded-wait test hook; only the bounds-checked debug build
    (libdopt_checked.so) has it."""
    if "dopt_debug_starve_copy" not in _c:
        raise DoptError(E_INVALID, "dopt_debug_starve_copy: only the bounds-checked debug build has this hook")
    _check(_c["dopt_debug_starve_copy"](tile))


def dopt_debug_bounds_record():
    """(failed checks, first site, first element, extent) of a bounds-checked
    build's record on the current device, which the call clears."""
    out = (_I64 * 4)()
    _check(_c["dopt_debug_bounds_record"](out))
    return tuple(out)


def dopt_kernel_launches():
    return int(_c["dopt_kernel_launches"]())


def dopt_memory_ledger(P, N, stage):
    parts = (_I64 * 5)()
    total = _check(_c["dopt_memory_ledger"](P, N, stage, parts))
    return total, list(parts)


def dopt_comm_bytes(P, N, elem_bytes, kind):
    return _check(_c["dopt_comm_bytes"](P, N, elem_bytes, kind))


def dopt_loss_scaler_init(initial_scale=2.0**16, growth_factor=2.0, backoff_factor=0.5,
                          growth_interval=1000, hysteresis=1, min_scale=1.0):
    s = dopt_loss_scaler()
    _check(_c["dopt_loss_scaler_init"](ctypes.byref(s), initial_scale, growth_factor,
                                       backoff_factor, growth_interval, hysteresis, min_scale))
    return s


def dopt_loss_scaler_update(s, found_inf):
    _check(_c["dopt_loss_scaler_update"](ctypes.byref(s), int(bool(found_inf))))
    return s.scale


def exported_symbols():
    """Names of the C entry points this binding resolved in the library."""
    return sorted(_c)


__all__ = [n for n in dir() if n.startswith("dopt_")] + [
    "ShardMap", "StepArgs", "DoptError", "exported_symbols"]
