#!/usr/bin/env python
"""Benchmark of the sharded mixed-precision Adam step (ZeRO-1 / Megatron
DistributedOptimizer) on GB300.

One step = the whole hot path over one rank's shard of the Llama-7B-shaped
workload: the emulated reduce-scatter of 8 fp32 replica grads, prepare_grads
(unscale, inf/NaN), the global grad norm and clip, AdamW on the fp32 master /
m / v, and the bf16 write-back into the param buffer -- through the
library's C ABI (dopt_step), inputs resident in HBM.

Prints ONE JSON line on rank 0.  Usage:
  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 launch under torch.distributed.run: every rank runs an independent
replica of the workload on its own GPU (the emulated DP ranks live inside one
GPU, so the path has no cross-GPU exchange); value = all ranks' elements /
the slowest rank's time.

--impl reference times the CPU oracle (a plain scalar C restatement of the
pages' arithmetic) on the host cores, on a bounded sample of the same
workload.  The oracle is test infrastructure; this leg and the cpu_baseline
key are the only places bench.py runs it.
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sharded Adam step params/s and HBM GB/s (% of GB300 peak), 1 GPU"
UNIT = "params/s"
DEFAULT_WORKLOAD = "llama_7b_dp8_rank0"
# the other configurations of the method's workloads: the toy MLP, GPT-2
# small, Llama-1.3B fp16, and the Llama-7B 2 x 8 hierarchy at 40M buckets
OTHER_CONFIGS = "toy_mlp_dp4,gpt2_small_dp8,llama_1p3b_fp16_dp8,llama_7b_dp16_2x8_40m"
CPU_SAMPLE_ELEMENTS = 32 * 2**20
F32, BF16, F16 = 0, 1, 2
ELEM_BYTES = {F32: 4, BF16: 2, F16: 2}
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, vendor nominal (context beside the measured copy peak)
STATS_BYTES = 40  # sizeof(dopt_step_stats): the step's results read back to the host


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--layers", type=int, default=None,
                   help="override the layer count (a smaller case of the same kernels)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--check-grads", action="store_true",
                   help="turn on the pre-reduction grad check (largest |g| per replica and bucket)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=5)
    p.add_argument("--other-configs", default=OTHER_CONFIGS,
                   help="comma-separated workloads also timed (N=1 only) after the main one, "
                        "each reported under other_configs; empty: none")
    p.add_argument("--graph", action="store_true",
                   help="time the step replayed from a CUDA graph (device step counter) "
                        "against dopt_step calls")
    p.add_argument("--staged", action="store_true",
                   help="time the bucket-staged step against the fused step, with the grads "
                        "produced bucket by bucket by a stand-in for the backward pass")
    p.add_argument("--multirank", action="store_true",
                   help="time two ranks of the workload's instance on this GPU, their norm "
                        "statistics combined through the host, on the device, or on the device "
                        "inside one CUDA graph")
    return p.parse_args(argv)


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def workload_config(name, layers=None):
    from synth import workloads as W
    cfg = W.config(name)
    if layers is not None:
        cfg["params"] = W.llama(layers, 4096, 11008, 32000)
        cfg["name"] = f"{name}_{layers}layers"
    return cfg


SHAPES = {
    "toy_mlp_dp4": "toy MLP, 4 x {W [1024,512], b [1024], W2 [512,1024], b2 [512]}",
    "gpt2_small_dp8": "GPT-2-small-shaped (12 layers, d=768, ffn 3072, vocab 50257), fp32 LayerNorm group",
    "llama_1p3b_fp16_dp8": "Llama-1.3B-shaped (24 layers, d=2048, ffn 5504, vocab 32000), fp16 params, "
                           "fp32 RMSNorm group, loss scale 65536",
}


def describe(cfg, n_elems):
    n_rep = cfg["dp"] * cfg["n_inst"]
    gtype = "fp32" if cfg["grad_reduce_in_fp32"] else "16-bit"
    if cfg["ranks"] == "all":
        who = f"all {cfg['dp']} ranks' shards ({n_elems} param elements)"
        reps = f"{n_rep} {gtype} replica grad buffers (whole buffers)"
    else:
        who = f"rank {cfg['ranks'][0]}'s shard of {n_elems} param elements"
        reps = f"{n_rep} {gtype} replica grad shards"
    base = cfg["name"].split("_2layers")[0]
    shape = SHAPES.get(base)
    if shape is None:
        n_layers = sum(1 for p in cfg["params"] if p["name"].endswith("q_proj"))
        shape = (f"Llama-7B-shaped ({n_layers} layers, d=4096, ffn 11008, vocab 32000), bf16 params + "
                 f"fp32 RMSNorm group")
    avg = ", averaged in the collective" if cfg.get("average") else ""
    return (f"{cfg['name']}: {shape}, DP={cfg['dp']} x {cfg['n_inst']} instance(s) emulated, {who}, "
            f"{reps}{avg}, bucket {cfg['bucket_size']}, AdamW lr 1e-4 betas (0.9, 0.95) eps 1e-8 "
            f"wd 0.1, clip 1.0")


def algorithmic_bytes(D, pm, n_rep, ranks):
    """Per-stage algorithmic DRAM bytes of one step and the stepped element count.
    K1 reads every replica element once and writes the main grad once (fp32,
    or for 16-bit grads the reduced grad in the grad dtype); K3 reads that
    main grad, master, m, v once and writes master, m, v and (16-bit buffers)
    the param once.  The fp32 buffer's master is its param buffer."""
    k1 = k3 = elems = 0
    for b in range(D.dopt_num_buffers(pm)):
        info = D.dopt_buffer_info_get(pm, b)
        n = sum(s["gbuf_local"][1] - s["gbuf_local"][0]
                for r in ranks for s in D.dopt_rank_shards(pm, b, r))
        elems += n
        g = ELEM_BYTES[info["grad_dtype"]]  # the main grad between the passes takes g bytes too
        k1 += n * (n_rep * g + g)
        k3 += n * (g + 12 + 12 + (ELEM_BYTES[info["param_dtype"]] if info["param_dtype"] != F32 else 0))
    return k1, k3, elems


def line_config(cfg, elements, rep_bytes, l2_bytes, check_grads):
    """The `config` object of both arms' lines: the workload, its stepped
    elements and replicas, how L2 is kept out of the timing, the
    parallelism and the grad check."""
    if l2_bytes is None:
        l2 = "L2 size unknown (no GPU visible)"
    elif rep_bytes < 2 * l2_bytes:
        l2 = (f"inputs smaller than L2 ({rep_bytes / 1e6:.1f} MB of replica grads): "
              f"{2 * l2_bytes / 1e6:.0f} MB written, then another {2 * l2_bytes / 1e6:.0f} MB read, "
              "between timed steps (L2 holds neither the step's inputs nor dirty lines of the "
              "flush), each step timed from its first to its last event")
    else:
        l2 = ("no flush needed: inputs larger than L2 (the replica grads alone are "
              f"{rep_bytes / 1e9:.1f} GB per step)")
    return {"workload": describe(cfg, elements), "elements_per_step": elements,
            "replicas": cfg["dp"] * cfg["n_inst"], "l2": l2,
            "parallelism": "replicas only: each GPU runs its own emulated DP instance",
            "grad_check": bool(check_grads)}


def oracle_counts(cfg):
    """Stepped elements and replica-grad bytes of one step, counted from the
    oracle's shard map (the reference arm's path: no product code)."""
    import oracle
    m = oracle.ShardMap(cfg["params"], cfg["dp"], cfg["bucket_size"], cfg["grad_reduce_in_fp32"])
    ranks = list(range(cfg["dp"])) if cfg["ranks"] == "all" else list(cfg["ranks"])
    n_rep = cfg["dp"] * cfg["n_inst"]
    elements = rep_bytes = 0
    for bi, buf in enumerate(m.buffers):
        elements += sum(v["gbuf_local"].size for r in ranks for _, _, v in m.rank_pieces(bi, r))
        n = buf.numel if cfg["layout"] == "full" else m.shard_numel(bi)
        rep_bytes += n_rep * n * ELEM_BYTES[buf.grad_dtype]
    return elements, rep_bytes


def read_once_bytes(D, pm, n_rep, ranks):
    """Bytes of one step if every input were read once and every output
    written once, with no main grad between two passes: the replica grads,
    master, m and v read; master, m, v and (16-bit buffers) the param
    written.  A global-norm clip cannot reach it (the update of any element
    needs every element's grad first), so it is reported beside the
    two-pass count, not as the target."""
    total = 0
    for b in range(D.dopt_num_buffers(pm)):
        info = D.dopt_buffer_info_get(pm, b)
        n = sum(s["gbuf_local"][1] - s["gbuf_local"][0]
                for r in ranks for s in D.dopt_rank_shards(pm, b, r))
        p = ELEM_BYTES[info["param_dtype"]] if info["param_dtype"] != F32 else 0
        total += n * (n_rep * ELEM_BYTES[info["grad_dtype"]] + 24 + p)
    return total


class Workload:
    """Device tensors of one rank's shard, filled by the seeded generator."""

    def __init__(self, cfg):
        import torch
        import synth
        import mixed_precision_adam_gb300 as D
        self.D, self.torch, self.cfg = D, torch, cfg
        self.all_ranks = cfg["ranks"] == "all"
        self.ranks = list(range(cfg["dp"])) if self.all_ranks else list(cfg["ranks"])
        self.rank = D.ALL_RANKS if self.all_ranks else self.ranks[0]
        self.full = cfg["layout"] == "full"
        self.n_rep = cfg["dp"] * cfg["n_inst"]
        self.pm = D.dopt_build_shard_map(cfg["params"], cfg["dp"], cfg["bucket_size"],
                                         cfg["grad_reduce_in_fp32"], False)
        dev = torch.device("cuda")
        stream = torch.cuda.current_stream().cuda_stream
        pkey = synth.key(cfg["seed"], synth.STREAM_PARAM, 0, 0)
        kinds = {F32: synth.OUT_F32, BF16: synth.OUT_BF16, F16: synth.OUT_F16}
        tdt = {F32: torch.float32, BF16: torch.int16, F16: torch.int16}
        self.reps, self.main, self.master, self.m, self.v, self.params = [], [], [], [], [], []
        for b in range(D.dopt_num_buffers(self.pm)):
            info = D.dopt_buffer_info_get(self.pm, b)
            S = info["shard_numel"]
            n_local = S * len(self.ranks)
            buckets = [D.dopt_bucket_info_get(self.pm, b, k) for k in range(info["n_buckets"])]
            reps = []
            for k in range(self.n_rep):
                gkey = synth.key(cfg["seed"], synth.STREAM_GRAD, 1, k)
                if self.full:
                    t = torch.empty(info["numel"], dtype=tdt[info["grad_dtype"]], device=dev)
                    synth.cuda_normal_(t.data_ptr(), info["numel"], gkey, 0, cfg["grad_sigma"],
                                       kinds[info["grad_dtype"]], stream)
                else:
                    t = torch.empty(S, dtype=tdt[info["grad_dtype"]], device=dev)
                    for bk in buckets:
                        s = bk["shard_numel"]
                        synth.cuda_normal_(t.data_ptr() + bk["shard_base"] * t.element_size(), s,
                                           gkey, bk["offset"] + self.ranks[0] * s, cfg["grad_sigma"],
                                           kinds[info["grad_dtype"]], stream)
                reps.append(t)
            self.reps.append(reps)
            p = torch.empty(info["numel"], dtype=tdt[info["param_dtype"]], device=dev)
            synth.cuda_normal_(p.data_ptr(), info["numel"], pkey, 0, cfg["param_sigma"],
                               kinds[info["param_dtype"]], stream)
            self.params.append(p)
            if info["param_dtype"] == F32:
                self.master.append(None)
            else:
                mt = torch.empty(n_local, dtype=torch.float32, device=dev)
                vk = synth.OUT_F32_OF_BF16 if info["param_dtype"] == BF16 else synth.OUT_F32_OF_F16
                for slot, r in enumerate(self.ranks):
                    for bk in buckets:
                        s = bk["shard_numel"]
                        synth.cuda_normal_(mt.data_ptr() + (slot * S + bk["shard_base"]) * 4, s, pkey,
                                           bk["offset"] + r * s, cfg["param_sigma"], vk, stream)
                self.master.append(mt)
            self.m.append(torch.zeros(n_local, dtype=torch.float32, device=dev))
            self.v.append(torch.zeros(n_local, dtype=torch.float32, device=dev))
            self.main.append(torch.empty(n_local, dtype=torch.float32, device=dev))
        self.ws_bytes = D.dopt_workspace_bytes(self.pm, self.rank)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()
        self.k1_bytes, self.k3_bytes, self.elements = algorithmic_bytes(D, self.pm, self.n_rep,
                                                                        self.ranks)
        self.read_once_bytes = read_once_bytes(D, self.pm, self.n_rep, self.ranks)
        self.t_applied = 0

    def args(self, reps=None):
        D = self.D
        return D.StepArgs(self.pm, self.rank, reps or self.reps, self.main, self.master, self.m,
                          self.v, self.params, self.cfg["hp"], self.t_applied + 1, self.ws,
                          self.ws_bytes, n_instances=self.cfg["n_inst"],
                          layout=D.LAYOUT_FULL_BUFFER if self.full else D.LAYOUT_SHARD_ONLY,
                          average_in_collective=self.cfg.get("average", False),
                          inv_loss_scale=1.0 / self.cfg["loss_scale"], max_norm=self.cfg["max_norm"],
                          stream=self.torch.cuda.current_stream())

    def step(self, args, events=None):
        args.set_step(self.t_applied + 1)
        args.set_stage_events(events)
        found, norm = self.D.dopt_step(args)
        if not found:
            self.t_applied += 1
        return found, norm


class ClockSampler:
    """nvidia-smi clock / throttle samples every 200 ms while running."""

    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.samples.append(parts)

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self):
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[1]) for s in self.samples if num(s[1]) is not None]
        mx = [num(s[2]) for s in self.samples if num(s[2]) is not None]
        reasons = set()
        for s in self.samples:
            for name, v in zip(["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                "sw_power_cap"], s[5:9]):
                if v.lower() in ("active", "1"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(self.samples)}


REJECTED_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def clocks_rejected(clk, low=0.85):
    """A timed region's clock record that does not count: a hardware or
    thermal slowdown was active, or the median SM clock sat below `low` x
    its maximum with no reason active (a clock lock).  sw_power_cap alone
    is kept."""
    if any(r in clk["reasons"] for r in REJECTED_REASONS):
        return True
    sm, mx = clk.get("sm_mhz"), clk.get("sm_max_mhz")
    return bool(sm and mx and sm < low * mx and not clk["reasons"])


def any_rank(flag, world):
    """True on every rank when `flag` is true on any rank."""
    if world <= 1:
        return bool(flag)
    import torch
    import torch.distributed as dist
    t = torch.tensor([1.0 if flag else 0.0], dtype=torch.float64)
    if dist.get_backend() == "nccl":
        t = t.cuda()
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return bool(t.item() > 0)


def host_available_bytes():
    """MemAvailable of /proc/meminfo (bytes); a large value when unknown."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 1 << 50


def measured_peak_hbm():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


K1_SOURCES = ("kernels.cuh", "tma.cuh", "k1.cuh", "k1_f32.cu")


def code_of(text):
    """C/C++ source without comments and with whitespace runs collapsed:
    what a change must touch to change the compiled kernel."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def k1_source_sha256():
    """sha256 over the code (comments and layout removed) of the sources of
    the fp32 reduce/prepare kernel, in order."""
    h = hashlib.sha256()
    for f in K1_SOURCES:
        with open(os.path.join(ROOT, "mixed_precision_adam_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(code_of(fh.read()).encode())
    return h.hexdigest()


def k1_variant(cfg, check_grads):
    """What selects the reduce/prepare kernel of a workload's bf16 buffer:
    replicas per instance, instances, grad dtype, replica layout, averaging
    and the grad check."""
    return {"replicas": cfg["dp"], "instances": cfg["n_inst"],
            "grad_dtype": "f32" if cfg["grad_reduce_in_fp32"] else "16-bit",
            "layout": cfg["layout"], "average": bool(cfg.get("average", False)),
            "grad_check": bool(check_grads)}


def recorded_traffic(elements_k1, variant):
    """DRAM traffic of the reduce/prepare pass from the committed ncu summary
    (taken on a small case of the same kernel), scaled per element to this
    launch's elements; None when the kernel source changed since the
    counters were taken, or when this workload runs another variant of the
    kernel than the one captured."""
    path = os.path.join(ROOT, "profiles", "ncu_k1_traffic.json")
    try:
        rec = json.load(open(path))
    except (OSError, ValueError):
        return None
    if k1_source_sha256() != rec.get("source_sha256") or rec.get("variant") != variant:
        return None
    return rec["dram_bytes_per_element"] * elements_k1


class OracleSample:
    """A fixed sample of the workload for the CPU oracle: the first `elements`
    elements of the selected rank's shard of the bf16 buffer, with its replica
    grads and state in host memory.  step() runs one full oracle step over it
    (reduce, prepare, sum of squares, clip coefficient, AdamW, RNE cast),
    single-threaded."""

    def __init__(self, cfg, elements):
        import ctypes
        import numpy as np
        import oracle
        import synth
        self.ctypes, self.oracle = ctypes, oracle
        om = oracle.ShardMap(cfg["params"], cfg["dp"], cfg["bucket_size"], cfg["grad_reduce_in_fp32"])
        self.cfg = cfg
        self.rank = 0 if cfg["ranks"] == "all" else cfg["ranks"][0]
        self.n_rep = cfg["dp"] * cfg["n_inst"]
        pieces, total = [], 0
        for pid, b, v in om.rank_pieces(0, self.rank):
            take = min(v["gbuf_local"].size, elements - total)
            if take <= 0:
                break
            pieces.append((pid, v["gbuf_world"].start, take))
            total += take
        self.pieces, self.elements = pieces, total
        buf = om.buffers[0]
        self.gdt, self.pdt = buf.grad_dtype, buf.param_dtype
        gkind = {F32: synth.OUT_F32, BF16: synth.OUT_BF16, F16: synth.OUT_F16}[self.gdt]
        self.reps = [np.concatenate([synth.normal(n, synth.key(cfg["seed"], synth.STREAM_GRAD, 1, k),
                                                  w, cfg["grad_sigma"], gkind) for _, w, n in pieces])
                     for k in range(self.n_rep)]
        pkey = synth.key(cfg["seed"], synth.STREAM_PARAM, 0, 0)
        mkind = {F32: synth.OUT_F32, BF16: synth.OUT_F32_OF_BF16, F16: synth.OUT_F32_OF_F16}[self.pdt]
        self.master = np.concatenate([synth.normal(n, pkey, w, cfg["param_sigma"], mkind)
                                      for _, w, n in pieces])
        self.m = np.zeros(total, np.float32)
        self.v = np.zeros(total, np.float32)
        self.out = np.zeros(total, np.uint16 if self.pdt != F32 else np.float32)
        self.main = np.zeros(total, np.float32)
        self.inv_scale = float(np.float32(1.0 / cfg["loss_scale"]))
        self.L = oracle.lib()
        self.arr = (ctypes.c_void_p * self.n_rep)(*[x.ctypes.data for x in self.reps])
        self.h = oracle.Hparams(**cfg["hp"])
        self.t = 0

    def _reduce(self, lo, hi):
        c, L = self.ctypes, self.L
        bad = L.or_reduce_prepare_run(self.arr, self.n_rep, self.cfg["n_inst"], self.gdt,
                                      int(bool(self.cfg.get("average", False))), lo,
                                      hi - lo, c.c_float(1.0), c.c_float(self.inv_scale),
                                      self.main.ctypes.data + 4 * lo)
        return bad, L.or_sumsq_run(self.main.ctypes.data + 4 * lo, hi - lo)

    def _adamw(self, lo, hi, coef, clip):
        c = self.ctypes
        self.L.or_adamw_run(self.main.ctypes.data + 4 * lo, hi - lo, coef, clip,
                            self.master.ctypes.data + 4 * lo, self.m.ctypes.data + 4 * lo,
                            self.v.ctypes.data + 4 * lo, c.byref(self.h), 1.0, self.t,
                            self.out.ctypes.data + self.out.itemsize * lo, self.pdt)

    def step(self, pool=None, threads=1):
        """One oracle step over the sample: on one thread, or on `threads`
        fixed chunks run by a thread pool (the C oracle runs without the
        GIL), the chunks' sums of squares added in chunk order."""
        c = self.ctypes
        step = -(-self.elements // threads)
        chunks = [(lo, min(self.elements, lo + step)) for lo in range(0, self.elements, step)]
        run = (lambda f, args: [f(*a) for a in args]) if pool is None else \
            (lambda f, args: list(pool.map(lambda a: f(*a), args)))
        parts = run(self._reduce, chunks)
        bad = sum(p[0] for p in parts)
        sumsq = 0.0
        for p in parts:
            sumsq += p[1]
        norm, coef = c.c_double(), c.c_double()
        clip = self.L.or_clip_coef(sumsq, self.cfg["max_norm"], c.byref(norm), c.byref(coef))
        if bad == 0:
            self.t += 1
            run(self._adamw, [(lo, hi, coef.value, clip) for lo, hi in chunks])

    def describe(self):
        names = {F32: "fp32", BF16: "bf16", F16: "fp16"}
        return (f"{self.elements} elements ({len(self.pieces)} param pieces) at the start of rank "
                f"{self.rank}'s {names[self.pdt]} shard of {self.cfg['name']}, {self.n_rep} "
                f"{names[self.gdt]} replicas")


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def time_oracle(sample, seconds_target, max_passes, threads):
    """Repeated full oracle steps on the sample for at least seconds_target
    seconds (at most max_passes): (passes, seconds)."""
    from concurrent.futures import ThreadPoolExecutor
    pool = ThreadPoolExecutor(threads) if threads > 1 else None
    try:
        passes, t0 = 0, time.perf_counter()
        while True:
            sample.step(pool, threads)
            passes += 1
            el = time.perf_counter() - t0
            if el >= seconds_target or passes >= max_passes:
                return passes, el
    finally:
        if pool is not None:
            pool.shutdown()


def cpu_baseline(cfg, seconds_target=8.0, max_passes=40):
    """The oracle timed on the host over a bounded sample of
    CPU_SAMPLE_ELEMENTS elements: on every host core (fixed chunks, one per
    core, the norm's partial sums added in chunk order) -- the reported value
    -- and on one thread."""
    sample = OracleSample(cfg, CPU_SAMPLE_ELEMENTS)
    cores = host_cores()
    p1, e1 = time_oracle(sample, seconds_target, max_passes, 1)
    pn, en = time_oracle(sample, seconds_target / 2, max_passes * cores, cores)
    return {"value": sample.elements * pn / en, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{sample.describe()}: {pn} full oracle steps in {en:.1f} s on {cores} threads "
                      f"(one chunk per thread); one thread: {p1} steps in {e1:.1f} s",
            "value_one_thread": sample.elements * p1 / e1}


# oracle elements per reference run: about 6 s on 16 host cores (about 90 s
# on one), so each step's sample stays a sizeable slice of the workload
REFERENCE_BUDGET_ELEMENTS = 3_000_000_000


def run_reference(args):
    rank, _, _ = dist_env()
    if rank != 0:
        return 0
    cfg = workload_config(args.workload, args.layers)
    # the same config object as this workload's line of the GPU arm
    elements, rep_bytes = oracle_counts(cfg)
    l2_bytes = None
    try:
        import torch
        if torch.cuda.is_available():
            l2_bytes = torch.cuda.get_device_properties(0).L2_cache_size
    except ImportError:
        pass
    per_step = REFERENCE_BUDGET_ELEMENTS // max(1, args.steps + args.warmup)
    per_step = max(1 << 20, min(CPU_SAMPLE_ELEMENTS, per_step))
    sample = OracleSample(cfg, per_step)
    cores = host_cores()
    from concurrent.futures import ThreadPoolExecutor
    pool = ThreadPoolExecutor(cores) if cores > 1 else None
    for _ in range(args.warmup):
        sample.step(pool, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        sample.step(pool, cores)
    el = time.perf_counter() - t0
    if pool is not None:
        pool.shutdown()
    value = sample.elements * args.steps / el
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "impl": "reference",
            "config": line_config(cfg, elements, rep_bytes, l2_bytes, False),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"each step: {sample.describe()}, {cores} threads "
                                       "(one fixed chunk each)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def aggregate(elapsed_ms, elements_per_step, steps, world):
    """Whole-job value: every rank's elements over the slowest rank's time."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([elapsed_ms], dtype=torch.float64)
    if world > 1:
        if dist.get_backend() == "nccl":
            t = t.cuda()
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    slowest = float(t.item())
    return elements_per_step * steps * world / (slowest / 1e3), slowest


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def timed_region(wl, sargs, steps, traced, local_rank, world):
    """One device-resident timed region of `steps` steps of workload wl:
    (elapsed ms, per-step events, kernel launches, clocks).  Untraced, each
    step records only the events before and after it; traced, all four
    stage events.  Inputs smaller than twice L2 get an L2 flush (a write,
    then a read of another buffer as large) between the steps, outside the
    timed work."""
    import torch
    D = wl.D
    l2_bytes = torch.cuda.get_device_properties(local_rank).L2_cache_size
    rep_bytes = sum(r.numel() * r.element_size() for reps in wl.reps for r in reps)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for e4 in ev:  # torch creates the CUDA event on its first record
        for e in e4:
            e.record()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    flush = torch.empty(2 * l2_bytes, dtype=torch.uint8, device="cuda") if rep_bytes < 2 * l2_bytes else None
    # after the write, a read of another buffer as large: L2 is left
    # holding clean lines, so the step does not pay the write-back of
    # the flush's own dirty lines
    clean = torch.zeros(2 * l2_bytes // 8, dtype=torch.int64, device="cuda") if flush is not None else None
    clocks = ClockSampler(local_rank)
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    launches0 = D.dopt_kernel_launches()
    start.record()
    for i in range(steps):
        if flush is not None:
            flush.fill_(i & 0xFF)
            clean.sum()
        wl.step(sargs, ev[i] if traced else [ev[i][0], None, None, ev[i][3]])
    end.record()
    torch.cuda.synchronize()
    barrier(world)
    launches = D.dopt_kernel_launches() - launches0
    clocks.stop()
    if flush is None:
        elapsed = start.elapsed_time(end)
    else:
        elapsed = sum(e[0].elapsed_time(e[3]) for e in ev)
    return elapsed, ev, launches, clocks.summary()


def measured(wl, sargs, steps, traced, local_rank, world, rank):
    """timed_region, taken once more when its clocks show a hardware or
    thermal slowdown, or SM clocks held well below their maximum with no
    reason given (a clock lock left behind); every rank decides alike.
    Returns (the region, the first attempt's clocks or None)."""
    out = timed_region(wl, sargs, steps, traced, local_rank, world)
    if any_rank(clocks_rejected(out[3]), world):
        log(f"[bench] rank {rank}: timed region taken again (clocks {out[3]})")
        return timed_region(wl, sargs, steps, traced, local_rank, world), out[3]
    return out, None


def other_config(name, args, local_rank):
    """One more workload timed like the main line's (device-resident step,
    an untraced and a traced region of the same steps, L2 flushed between
    steps when its inputs are smaller than twice L2), for the line's
    `other_configs`.  Never raises: a failure is reported in the entry."""
    import torch
    out = {"workload": name}
    try:
        cfg = workload_config(name)
        wl = Workload(cfg)
        sargs = wl.args()
        for _ in range(max(3, args.warmup)):
            wl.step(sargs)
        torch.cuda.synchronize()
        steps = max(5, min(args.steps, 50))
        (elapsed, _, launches, clk), first = measured(wl, sargs, steps, False, local_rank, 1, 0)
        (_, sev, _, sclk), _ = measured(wl, sargs, steps, True, local_rank, 1, 0)
        peak, _ = measured_peak_hbm()
        ms = elapsed / steps
        k1 = statistics.mean(e[0].elapsed_time(e[1]) for e in sev)
        k3 = statistics.mean(e[2].elapsed_time(e[3]) for e in sev)
        l2_bytes = torch.cuda.get_device_properties(local_rank).L2_cache_size
        rep_bytes = sum(r.numel() * r.element_size() for reps in wl.reps for r in reps)
        out.update({
            "config": line_config(cfg, wl.elements, rep_bytes, l2_bytes, False),
            "value": wl.elements / (ms * 1e-3), "unit": UNIT, "steps": steps,
            "ms_per_step": ms,
            "hbm_frac": (wl.k1_bytes + wl.k3_bytes) / (ms * 1e-3) / 1e9 / peak,
            "reduce_prepare_ms": k1, "reduce_prepare_frac": wl.k1_bytes / (k1 * 1e-3) / 1e9 / peak,
            "adamw_ms": k3, "adamw_frac": wl.k3_bytes / (k3 * 1e-3) / 1e9 / peak,
            "traced_ms_per_step": statistics.mean(e[0].elapsed_time(e[3]) for e in sev),
            "gpu_launches": launches, "clocks": clk, "stage_clocks": sclk})
        if first is not None:
            out["remeasured"] = {"first_clocks": first}
        del wl, sargs
    except Exception as e:  # reported, so the main line still prints
        out["error"] = f"{type(e).__name__}: {e}"[:300]
    try:
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    except Exception as e:
        out.setdefault("error", f"{type(e).__name__}: {e}"[:300])
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist
    rank, local_rank, world = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    import mixed_precision_adam_gb300 as D
    cfg = workload_config(args.workload, args.layers)
    wl = Workload(cfg)
    log(f"[bench] rank {rank}: {wl.elements} elements per step, workspace {wl.ws_bytes} B")
    sargs = wl.args()
    if args.check_grads:
        amax = torch.zeros((wl.n_rep, D.dopt_total_buckets(wl.pm)), dtype=torch.float32, device="cuda")
        sargs.set_grad_check(amax)
    for _ in range(args.warmup):
        wl.step(sargs)
    torch.cuda.synchronize()

    # device-resident timed region.  Inputs smaller than L2 (the toy MLP):
    # write a buffer of twice the L2 size between the timed steps and time
    # each step from the event before it to the event after it, so the
    # flushes stay outside the timed work.  The step is timed as a caller runs it, with
    # events before and after it only: a timing event recorded between the
    # reduce pass and the AdamW pass waits for the reduce grid to drain and
    # stops the AdamW CTAs from starting early (about 6 us a step on the toy
    # MLP, within the noise of the larger steps).  The per-pass durations come
    # from a second region of the same steps with all four stage events.
    l2_bytes = torch.cuda.get_device_properties(local_rank).L2_cache_size
    rep_bytes = sum(r.numel() * r.element_size() for reps in wl.reps for r in reps)

    (elapsed, ev, launches, clk), first_clocks = measured(wl, sargs, args.steps, False, local_rank, world, rank)
    (_, sev, _, sclk), first_sclocks = measured(wl, sargs, args.steps, True, local_rank, world, rank)
    k1 = statistics.mean(e[0].elapsed_time(e[1]) for e in sev)
    k2 = statistics.mean(e[1].elapsed_time(e[2]) for e in sev)
    k3 = statistics.mean(e[2].elapsed_time(e[3]) for e in sev)
    value, slowest = aggregate(elapsed, wl.elements, args.steps, world)

    peak, peak_src = measured_peak_hbm()
    k1_gbs = wl.k1_bytes / (k1 * 1e-3) / 1e9
    k3_gbs = wl.k3_bytes / (k3 * 1e-3) / 1e9
    step_gbs = (wl.k1_bytes + wl.k3_bytes) / (slowest / args.steps * 1e-3) / 1e9
    traffic = recorded_traffic(wl.elements, k1_variant(cfg, args.check_grads))

    # end to end: the step's inputs (the replica grads) copied in from pinned
    # host memory every step, then the C-ABI step, which reads back found_inf
    # and the norm
    e2e = None
    eargs = None
    if not args.no_e2e:
        # distinct pinned host copies of every replica, unless all ranks' copies
        # would take more than half of the host's available memory: then each
        # rank pins fewer host buffers and copies them into several replicas
        # (the bytes moved per step stay the same)
        per_rep = [r.numel() * r.element_size() for reps in wl.reps for r in reps]
        budget = 0.5 * host_available_bytes() / world
        host_reps, used = [], 0
        for reps in wl.reps:
            hb = []
            for k, r in enumerate(reps):
                nbytes = r.numel() * r.element_size()
                if used + nbytes <= budget or k == 0:
                    h = torch.empty_like(r, device="cpu", pin_memory=True)
                    h.copy_(r)
                    used += nbytes
                    hb.append(h)
                else:
                    hb.append(hb[k % len(hb)])
            host_reps.append(hb)
        # the C-ABI step with host replicas: the library copies each bucket's
        # replica slices on its copy stream and reduces the bucket as soon as
        # they land (dopt_step_from_host); it needs the bucket-staged workspace
        ws_b = D.dopt_workspace_bytes_bucketed(wl.pm, wl.rank)
        ws_staged = torch.empty(ws_b, dtype=torch.uint8, device="cuda")
        eargs = wl.args()
        eargs.c.workspace, eargs.c.workspace_bytes = ws_staged.data_ptr(), ws_b
        if args.check_grads:
            eargs.set_grad_check(amax)
        # bytes the library copies per step: every replica's part of each
        # bucket that the step reads
        h2d = 0
        for b in range(D.dopt_num_buffers(wl.pm)):
            info = D.dopt_buffer_info_get(wl.pm, b)
            for k in range(info["n_buckets"]):
                bk = D.dopt_bucket_info_get(wl.pm, b, k)
                n = bk["numel"] if (wl.full and wl.all_ranks) else bk["shard_numel"]
                h2d += n * ELEM_BYTES[info["grad_dtype"]] * wl.n_rep
        eargs.set_step(wl.t_applied + 1)  # one untimed step (creates the copy stream)
        if not D.dopt_step_from_host(eargs, host_reps)[0]:
            wl.t_applied += 1
        torch.cuda.synchronize()
        distinct = len({id(h) for hb in host_reps for h in hb})
        n_e2e = max(1, min(args.e2e_steps, args.steps))
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        e0.record()
        for _ in range(n_e2e):
            eargs.set_step(wl.t_applied + 1)
            found, _ = D.dopt_step_from_host(eargs, host_reps)
            if not found:
                wl.t_applied += 1
        e1.record()
        torch.cuda.synchronize()
        wall = (time.perf_counter() - t0) * 1e3
        barrier(world)
        e2e_value, _ = aggregate(max(e0.elapsed_time(e1), wall), wl.elements, n_e2e, world)
        del ws_staged
        note = ("replica grads copied from pinned host memory each step by dopt_step_from_host, "
                "bucket by bucket, each bucket reduced as soon as its copies land")
        if distinct < len(per_rep):
            note += f" ({distinct} distinct host buffers for {len(per_rep)} replicas: host memory bound)"
        e2e = {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": STATS_BYTES, "steps": n_e2e, "note": note}
        del host_reps

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0
    cpu = None if args.no_cpu_baseline else cpu_baseline(cfg)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": slowest / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": line_config(cfg, wl.elements, rep_bytes, l2_bytes, args.check_grads),
        "hbm_gbs": step_gbs, "hbm_frac": step_gbs / peak,
        "read_once_ideal": {"bytes_per_step": wl.read_once_bytes,
                            "ms_at_peak": wl.read_once_bytes / (peak * 1e9) * 1e3,
                            "step_frac": wl.read_once_bytes / (peak * 1e9) * 1e3 / (slowest / args.steps),
                            "note": "every input read once, no main grad between two passes: "
                                    "out of reach with a global-norm clip"},
        "roofline": {"bound": "hbm", "achieved": k1_gbs, "peak": peak, "unit": "GB/s",
                     "frac": k1_gbs / peak, "traffic": traffic, "kernel": "k1_reduce_prepare",
                     "algorithmic_bytes_per_launch": wl.k1_bytes, "peak_source": peak_src,
                     "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": k1_gbs / NOMINAL_HBM_GBS},
        "ms_per_step_median": statistics.median(e[0].elapsed_time(e[3]) for e in ev),
        "stages": {"reduce_prepare_ms": k1, "norm_finalize_ms": k2, "adamw_ms": k3,
                   "adamw_gbs": k3_gbs, "adamw_frac": k3_gbs / peak,
                   "step_bytes": wl.k1_bytes + wl.k3_bytes,
                   "traced_ms_per_step": statistics.mean(e[0].elapsed_time(e[3]) for e in sev),
                   "clocks": sclk,
                   "note": "per-pass times from a second timed region of the same steps with "
                           "events recorded between the passes; ms_per_step and value from "
                           "the region without them"},
        "e2e": e2e, "gpu_launches": launches, "clocks": clk, "cpu_baseline": cpu,
    }
    if first_clocks is not None or first_sclocks is not None:
        line["remeasured"] = {"first_clocks": first_clocks, "first_stage_clocks": first_sclocks}
    names = [n for n in args.other_configs.split(",") if n] if world == 1 else []
    if names:
        # the other workloads, each in turn on its own, after the main one is freed
        del sargs, wl, eargs
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        line["other_configs"] = [other_config(n, args, local_rank) for n in names]
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_staged(args):
    """Overlap of the per-bucket reduce with the production of the grads.

    Each step first produces the replica grads (the generator's fill kernel
    writing every replica's slice of a bucket stands in for the backward pass
    finishing that bucket), then steps.  Sequential: produce every bucket,
    then the fused step.  Staged: as soon as a bucket is produced, its
    reduce/prepare runs on a side stream; after the last bucket, the norm
    finalize, then AdamW and the write-back bucket by bucket in forward order
    (last bucket first)."""
    import torch
    import synth
    import mixed_precision_adam_gb300 as D
    cfg = workload_config(args.workload, args.layers)
    if cfg["layout"] != "shard":
        raise SystemExit("--staged takes a shard-layout workload")
    wl = Workload(cfg)
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    kinds = {F32: synth.OUT_F32, BF16: synth.OUT_BF16, F16: synth.OUT_F16}
    buckets = []
    for b in range(D.dopt_num_buffers(wl.pm)):
        info = D.dopt_buffer_info_get(wl.pm, b)
        for k in range(info["n_buckets"]):
            buckets.append((b, k, info, D.dopt_bucket_info_get(wl.pm, b, k)))

    def produce(b, k, info, bk):
        s = bk["shard_numel"]
        for r, t in enumerate(wl.reps[b]):
            synth.cuda_normal_(t.data_ptr() + bk["shard_base"] * t.element_size(), s,
                               synth.key(cfg["seed"], synth.STREAM_GRAD, 1, r),
                               bk["offset"] + wl.ranks[0] * s, cfg["grad_sigma"],
                               kinds[info["grad_dtype"]], main.cuda_stream)

    fused = wl.args()
    staged = wl.args()
    ws_b = D.dopt_workspace_bytes_bucketed(wl.pm, wl.rank)
    bws = torch.empty(ws_b, dtype=torch.uint8, device="cuda")
    staged.c.workspace, staged.c.workspace_bytes = bws.data_ptr(), ws_b

    def step_fused():
        for x in buckets:
            produce(*x)
        fused.set_step(wl.t_applied + 1)
        D.dopt_step_async(fused)

    def step_staged():
        staged.set_step(wl.t_applied + 1)
        staged.set_stream(side)
        for (b, k, info, bk) in buckets:
            produce(b, k, info, bk)
            ev = torch.cuda.Event()
            ev.record(main)
            side.wait_event(ev)
            D.dopt_step_reduce_buckets(staged, b, k, 1)
        done = torch.cuda.Event()
        done.record(side)
        main.wait_event(done)
        staged.set_stream(main)
        D.dopt_step_finalize(staged)
        for (b, k, info, bk) in reversed(buckets):
            D.dopt_step_update_buckets(staged, b, k, 1)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.steps

    t_fused = timed(step_fused)
    t_staged = timed(step_staged)
    line = {"metric": "grad production + step, fused vs bucket-staged (ms per step)",
            "workload": describe(cfg, wl.elements), "buckets": len(buckets),
            "steps": args.steps, "warmup": args.warmup,
            "produce_then_fused_ms": t_fused, "bucket_staged_overlapped_ms": t_staged,
            "saving_ms": t_fused - t_staged}
    print(json.dumps(line), flush=True)
    return 0


def run_multirank(args):
    """Ranks 0 and 1 of a shard-layout workload's instance, one after the other
    on this GPU, each through the bucket-staged entry points, their norm
    statistics combined three ways: read to the host and passed back as
    remote terms (a host round trip between the passes), combined on the
    device (dopt_step_local_stats, a device add and max, d_global_*), and the
    device form captured in one CUDA graph with device step counters.  The
    two ranks' sum stands in for the instance's all-reduce (timing only)."""
    import torch
    import mixed_precision_adam_gb300 as D
    cfg = workload_config(args.workload, args.layers)
    if cfg["layout"] != "shard":
        raise SystemExit("--multirank takes a shard-layout workload")
    ranks = []
    for r in (0, 1):
        wl = Workload(dict(cfg, ranks=[r]))
        wsb = D.dopt_workspace_bytes_bucketed(wl.pm, r)
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        a = wl.args()
        a.c.workspace, a.c.workspace_bytes = ws.data_ptr(), wsb
        ranks.append(dict(wl=wl, ws=ws, args=a, local=torch.zeros(1, dtype=torch.float64, device="cuda"),
                          flag=torch.zeros(1, dtype=torch.int32, device="cuda")))
    nbk = [[D.dopt_buffer_info_get(rk["wl"].pm, b)["n_buckets"] for b in range(D.dopt_num_buffers(rk["wl"].pm))]
           for rk in ranks]
    glob = torch.zeros(1, dtype=torch.float64, device="cuda")
    gflag = torch.zeros(1, dtype=torch.int32, device="cuda")

    def reduce_all():
        for rk, nb in zip(ranks, nbk):
            for b, n in enumerate(nb):
                D.dopt_step_reduce_buckets(rk["args"], b, 0, n)
            D.dopt_step_local_stats(rk["args"], rk["local"], rk["flag"])

    def update_all():
        for rk, nb in zip(ranks, nbk):
            D.dopt_step_finalize(rk["args"])
            for b, n in enumerate(nb):
                D.dopt_step_update_buckets(rk["args"], b, 0, n)

    def host_step():
        reduce_all()
        loc = [float(rk["local"].item()) for rk in ranks]  # the host round trip
        bad = [int(rk["flag"].item()) for rk in ranks]
        for i, rk in enumerate(ranks):
            rk["args"].set_global_stats(None, None)
            rk["args"].c.remote_sumsq, rk["args"].c.remote_found_inf = loc[1 - i], bad[1 - i]
        update_all()

    def device_step():
        reduce_all()
        torch.add(ranks[0]["local"], ranks[1]["local"], out=glob)
        torch.maximum(ranks[0]["flag"], ranks[1]["flag"], out=gflag)
        for rk in ranks:
            rk["args"].c.remote_sumsq, rk["args"].c.remote_found_inf = 0.0, 0
            rk["args"].set_global_stats(glob, gflag)
        update_all()

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.steps

    t_host = timed(host_step)
    t_dev = timed(device_step)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        for rk in ranks:
            rk["d_step"] = torch.zeros(1, dtype=torch.int64, device="cuda")
            rk["args"].set_device_step(rk["d_step"])
            rk["args"].set_stream(s)
        with torch.cuda.graph(graph, stream=s):
            device_step()
    torch.cuda.synchronize()
    t_graph = timed(graph.replay)
    line = {"metric": "two ranks' bucket-staged steps: norm statistics combined through the host vs on the "
                      "device vs on the device in one CUDA graph (ms per step of both ranks)",
            "workload": describe(cfg, ranks[0]["wl"].elements) + "; ranks 0 and 1, one after the other",
            "steps": args.steps, "warmup": args.warmup, "host_combined_ms": t_host,
            "device_combined_ms": t_dev, "device_graph_ms": t_graph,
            "elements_per_step": ranks[0]["wl"].elements + ranks[1]["wl"].elements}
    print(json.dumps(line), flush=True)
    return 0


def run_graph(args):
    """The fused step three ways: dopt_step calls (each waits for found_inf),
    dopt_step_async calls back to back, and one CUDA-graph replay per step
    (step counter in device memory, no host work between steps)."""
    import torch
    import mixed_precision_adam_gb300 as D
    cfg = workload_config(args.workload, args.layers)
    wl = Workload(cfg)
    sargs = wl.args()

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.steps

    t_sync = timed(lambda: wl.step(sargs))
    t_async = timed(lambda: D.dopt_step_async(sargs))
    d_step = torch.zeros(1, dtype=torch.int64, device="cuda")
    gargs = wl.args()
    gargs.set_device_step(d_step)
    D.dopt_step_async(gargs)  # warm-up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        gargs.set_stream(s)
        with torch.cuda.graph(graph, stream=s):
            D.dopt_step_async(gargs)
    torch.cuda.synchronize()
    t_graph = timed(graph.replay)
    line = {"metric": "fused step latency: dopt_step vs async vs CUDA-graph replay (ms per step)",
            "workload": describe(cfg, wl.elements), "steps": args.steps, "warmup": args.warmup,
            "dopt_step_ms": t_sync, "dopt_step_async_ms": t_async, "graph_replay_ms": t_graph,
            "elements_per_step": wl.elements}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.staged:
        return run_staged(args)
    if args.multirank:
        return run_multirank(args)
    if args.graph:
        return run_graph(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
