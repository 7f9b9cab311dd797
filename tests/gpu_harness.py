"""Builds one workload's seeded inputs for both sides -- the CPU oracle (numpy
arrays) and the CUDA library (torch device tensors) -- runs optimizer steps
on each, and compares the results element by element.

Tolerances (the parity bar set for this path): shard map and
found_inf bit-exact; fp32 master, m and v within 4 ulp or 1e-6 relative;
16-bit params within 1 ulp of their type; grad norm within 1e-5 relative.
The main grad (the reduced, unscaled fp32 gradient) follows the same fixed
summation order on both sides and must be bit-exact (a NaN matching any
NaN: IEEE 754 does not fix the payload of a NaN result).
"""

import numpy as np

import oracle
import synth

F32, BF16, F16 = 0, 1, 2
KIND = {F32: synth.OUT_F32, BF16: synth.OUT_BF16, F16: synth.OUT_F16}
VALUE_KIND = {BF16: synth.OUT_F32_OF_BF16, F16: synth.OUT_F32_OF_F16}
INF_BITS = {F32: np.float32(np.inf), BF16: np.uint16(0x7F80), F16: np.uint16(0x7C00)}


def dopt():
    import mixed_precision_adam_gb300 as m
    return m


class HostCase:
    """Seeded inputs of a workload for the selected ranks, as numpy arrays."""

    def __init__(self, cfg):
        D = dopt()
        self.cfg = cfg
        dp, bs = cfg["dp"], cfg["bucket_size"]
        self.om = oracle.ShardMap(cfg["params"], dp, bs, cfg["grad_reduce_in_fp32"],
                                  cfg["pad_for_high_busbw"])
        self.pm = D.dopt_build_shard_map(cfg["params"], dp, -1 if bs is None else bs,
                                         cfg["grad_reduce_in_fp32"], cfg["pad_for_high_busbw"])
        self.all_ranks = cfg["ranks"] == "all"
        self.ranks = list(range(dp)) if self.all_ranks else list(cfg["ranks"])
        self.rank_arg = D.ALL_RANKS if self.all_ranks else self.ranks[0]
        self.n_rep = dp * cfg["n_inst"]
        self.seed = cfg["seed"]
        self.params, self.state = [], []
        pkey = synth.key(self.seed, synth.STREAM_PARAM, 0, 0)
        for bi, buf in enumerate(self.om.buffers):
            S = self.om.shard_numel(bi)
            n_local = len(self.ranks) * S
            self.params.append(synth.normal(buf.numel, pkey, 0, cfg["param_sigma"],
                                            KIND[buf.param_dtype]))
            st = {"exp_avg": np.zeros(n_local, np.float32),
                  "exp_avg_sq": np.zeros(n_local, np.float32)}
            if cfg.get("warm_state"):
                st["exp_avg"] = self.to_local(bi, synth.normal(
                    buf.numel, synth.key(self.seed, synth.STREAM_EXP_AVG, 0, 0), 0, 1e-4))
                st["exp_avg_sq"] = self.to_local(bi, synth.uniform(
                    buf.numel, synth.key(self.seed, synth.STREAM_EXP_AVG_SQ, 0, 0), 0, 1e-7))
            if buf.param_dtype != F32:
                full = synth.normal(buf.numel, pkey, 0, cfg["param_sigma"],
                                    VALUE_KIND[buf.param_dtype])
                st["master"] = self.to_local(bi, full)
            self.state.append(st)
        self.t_applied = 0

    def to_local(self, bi, world):
        """Gathers a buffer-indexed array into the flat shard layout of the ranks."""
        S = self.om.shard_numel(bi)
        out = np.zeros(len(self.ranks) * S, dtype=world.dtype)
        for slot, r in enumerate(self.ranks):
            for b in range(len(self.om.buffers[bi].buckets)):
                rg = self.om.bucket_world_range(bi, b, r)
                base = slot * S + self.om.bucket_shard_base(bi, b)
                out[base:base + rg.size] = world[rg.start:rg.end]
        return out

    def piece_mask(self, bi):
        """True at the flat-shard positions that hold param elements."""
        S = self.om.shard_numel(bi)
        mask = np.zeros(len(self.ranks) * S, dtype=bool)
        for slot, r in enumerate(self.ranks):
            for _, _, v in self.om.rank_pieces(bi, r):
                lo = slot * S + v["shard_offset"]
                mask[lo:lo + v["gbuf_local"].size] = True
        return mask

    def inf_position(self):
        """(buffer 0, world index) of the injected non-finite grad: the first
        param element at or after numel_unpadded * frac."""
        spec = self.cfg["inf_at"]
        buf = self.om.buffers[0]
        target = int(buf.numel_unpadded * spec["buffer_frac"])
        best = None
        for pid in buf.params:
            s, e, _ = buf.index[pid]
            if e > target and e > s:
                w = max(s, target)
                if best is None or w < best:
                    best = w
        return best

    def grads(self, t):
        """Replica grads of step t per buffer (layout per the config)."""
        cfg = self.cfg
        out = []
        for bi, buf in enumerate(self.om.buffers):
            reps = []
            for k in range(self.n_rep):
                key = synth.key(self.seed, synth.STREAM_GRAD, t, k)
                if cfg["layout"] == "full":
                    reps.append(synth.normal(buf.numel, key, 0, cfg["grad_sigma"], KIND[buf.grad_dtype]))
                else:
                    full = synth.normal(buf.numel, key, 0, cfg["grad_sigma"], KIND[buf.grad_dtype])
                    reps.append(self.to_local(bi, full))
            out.append(reps)
        spec = cfg.get("inf_at")
        if spec and spec["step"] == t:
            w = self.inf_position()
            rep = out[0][spec["replica"]]
            if cfg["layout"] == "full":
                rep[w] = INF_BITS[self.om.buffers[0].grad_dtype]
            else:
                marker = np.zeros(self.om.buffers[0].numel, dtype=bool)
                marker[w] = True
                loc = np.nonzero(self.to_local(0, marker))[0]
                if len(loc):
                    rep[loc[0]] = INF_BITS[self.om.buffers[0].grad_dtype]
        return out

    def oracle_step(self, grads, t):
        cfg = self.cfg
        return oracle.step(self.om, self.ranks, grads, self.state, self.params, cfg["hp"], t,
                           inv_scale=float(np.float32(1.0 / cfg["loss_scale"])),
                           max_norm=cfg["max_norm"], layout=cfg["layout"], n_inst=cfg["n_inst"],
                           average=cfg["average"], remote_sumsq=cfg.get("remote_sumsq", 0.0),
                           remote_found_inf=cfg.get("remote_found_inf", False),
                           grad_scale=float(np.float32(cfg.get("grad_scale", 1.0))))


class DeviceCase:
    """The same inputs on the GPU, stepped through the library's C ABI."""

    # Every device buffer sits between two guard regions of GUARD_BYTES
    # filled with a canary pattern; check_guards() finds any write outside a
    # buffer (the pool has no memory checker, so the tests look themselves).
    GUARD_BYTES = 256
    CANARY = 0xA5

    def __init__(self, hc):
        import torch
        D = dopt()
        self.hc = hc
        self.torch = torch
        self.guarded = []
        self.params = [self._up(p) for p in hc.params]
        self.master = [self._up(st["master"]) if "master" in st else None for st in hc.state]
        self.exp_avg = [self._up(st["exp_avg"]) for st in hc.state]
        self.exp_avg_sq = [self._up(st["exp_avg_sq"]) for st in hc.state]
        self.main = [self._alloc(len(st["exp_avg"]), torch.float32).zero_() for st in hc.state]
        self.ws_bytes = D.dopt_workspace_bytes(hc.pm, hc.rank_arg)
        self.ws = self._alloc(self.ws_bytes, torch.uint8)

    def _alloc(self, n, dtype):
        """A device tensor of n elements between two canary-filled guards."""
        torch = self.torch
        es = torch.empty(0, dtype=dtype).element_size()
        g = self.GUARD_BYTES
        raw = torch.full((2 * g + n * es,), self.CANARY, dtype=torch.uint8, device="cuda")
        self.guarded.append((raw, n * es))
        return raw[g:g + n * es].view(dtype)

    def _up(self, a):
        src = self.torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a.copy())
        t = self._alloc(src.numel(), src.dtype)
        t.copy_(src)
        return t

    def check_guards(self):
        """True when no guard byte of any buffer has changed."""
        g = self.GUARD_BYTES
        for raw, nbytes in self.guarded:
            if not (bool((raw[:g] == self.CANARY).all()) and bool((raw[g + nbytes:] == self.CANARY).all())):
                return False
        return True

    def step_args(self, reps, t, stream=None):
        D = dopt()
        cfg = self.hc.cfg
        return D.StepArgs(self.hc.pm, self.hc.rank_arg, reps, self.main, self.master, self.exp_avg,
                          self.exp_avg_sq, self.params, cfg["hp"], t, self.ws, self.ws_bytes,
                          n_instances=cfg["n_inst"],
                          layout=D.LAYOUT_FULL_BUFFER if cfg["layout"] == "full" else D.LAYOUT_SHARD_ONLY,
                          average_in_collective=cfg["average"],
                          inv_loss_scale=float(np.float32(1.0 / cfg["loss_scale"])),
                          max_norm=cfg["max_norm"], remote_sumsq=cfg.get("remote_sumsq", 0.0),
                          remote_found_inf=cfg.get("remote_found_inf", False),
                          stream=stream if stream is not None else self.torch.cuda.current_stream(),
                          grad_scale=float(np.float32(cfg.get("grad_scale", 1.0))))

    def step(self, grads, t):
        reps = [[self._up(r) for r in g] for g in grads]
        args = self.step_args(reps, t)
        found, norm = dopt().dopt_step(args)
        return found, norm

    def step_separate(self, grads, t):
        """The same step through the separate entry points (A2, A3, A4, A5+A6)."""
        D = dopt()
        torch = self.torch
        cfg = self.hc.cfg
        reps = [[self._up(r) for r in g] for g in grads]
        s = torch.cuda.current_stream()
        layout = D.LAYOUT_FULL_BUFFER if cfg["layout"] == "full" else D.LAYOUT_SHARD_ONLY
        for bi in range(len(self.main)):
            D.dopt_grad_reduce_shard(self.hc.pm, bi, self.hc.rank_arg, reps[bi], cfg["n_inst"], layout,
                                     cfg["average"], self.main[bi], self.ws, self.ws_bytes, s)
            D.dopt_prepare_grads(self.hc.pm, bi, self.hc.rank_arg,
                                 float(np.float32(1.0 / cfg["loss_scale"])), self.main[bi], self.ws,
                                 self.ws_bytes, s)
        d_norm = torch.zeros(1, dtype=torch.float32, device="cuda")
        d_coef = torch.zeros(1, dtype=torch.float32, device="cuda")
        d_found = torch.zeros(1, dtype=torch.int32, device="cuda")
        D.dopt_grad_norm(self.hc.pm, self.hc.rank_arg, self.ws, self.ws_bytes,
                         cfg.get("remote_sumsq", 0.0), cfg.get("remote_found_inf", False),
                         cfg["max_norm"], d_norm, d_coef, d_found, s)
        for bi in range(len(self.main)):
            D.dopt_adam_step(self.hc.pm, bi, self.hc.rank_arg, self.main[bi], self.master[bi],
                             self.exp_avg[bi], self.exp_avg_sq[bi], self.params[bi], cfg["hp"], t,
                             d_coef, d_found, s)
        torch.cuda.synchronize()
        return bool(d_found.item()), float(d_norm.item())

    def download(self):
        def dn(t):
            if t is None:
                return None
            a = t.cpu().numpy()
            return a.view(np.uint16) if a.dtype == np.int16 else a
        return ([dn(p) for p in self.params], [dn(m) for m in self.master],
                [dn(m) for m in self.exp_avg], [dn(v) for v in self.exp_avg_sq],
                [dn(m) for m in self.main])


def staged_step(dc, reps, t, group, streams, grad_amax=None):
    """Buckets reduced in backward order (bucket 0 first) on side streams,
    each waiting on an event that marks its grads ready; finalize; updates in
    forward order (last bucket first)."""
    D = dopt()
    hc = dc.hc
    ws_bytes = D.dopt_workspace_bytes_bucketed(hc.pm, hc.rank_arg)
    if getattr(dc, "bws", None) is None or dc.bws.numel() < ws_bytes:
        dc.bws = dc.torch.empty(ws_bytes, dtype=dc.torch.uint8, device="cuda")
    args = dc.step_args(reps, t)
    if grad_amax is not None:
        args.set_grad_check(grad_amax)
    args.c.workspace = dc.bws.data_ptr()
    args.c.workspace_bytes = ws_bytes
    main = dc.torch.cuda.current_stream()
    ready = []
    for bi in range(len(hc.om.buffers)):
        nbk = len(hc.om.buffers[bi].buckets)
        for k0 in range(0, nbk, group):
            ev = dc.torch.cuda.Event()
            ev.record(main)  # "the grads of these buckets are ready"
            s = streams[(bi + k0) % len(streams)]
            s.wait_event(ev)
            args.set_stream(s)
            D.dopt_step_reduce_buckets(args, bi, k0, min(group, nbk - k0))
            done = dc.torch.cuda.Event()
            done.record(s)
            ready.append(done)
    for ev in ready:
        main.wait_event(ev)
    args.set_stream(main)
    d_found = dc.torch.zeros(1, dtype=dc.torch.int32, device="cuda")
    d_norm = dc.torch.zeros(1, dtype=dc.torch.float32, device="cuda")
    D.dopt_step_finalize(args, d_found, d_norm)
    for bi in range(len(hc.om.buffers)):
        for k in reversed(range(len(hc.om.buffers[bi].buckets))):
            D.dopt_step_update_buckets(args, bi, k, 1)
    dc.torch.cuda.synchronize()
    return bool(d_found.item()), float(d_norm.item())


# ----------------------------------------------------------------------------
# The pre-reduction grad check (largest |g| per replica and bucket)

def encode_grad(gdt, value):
    """value in the grad dtype's storage (float32, or 16-bit bits)."""
    v = np.float32(value)
    if gdt == F32:
        return v
    return (oracle.round_bf16(v) if gdt == BF16 else oracle.round_f16(v))[0]


def plant(hc, grads, bi, k, w, value):
    """Sets replica k's grad of buffer bi at buffer index w, in whichever
    layout the replicas use."""
    enc = encode_grad(hc.om.buffers[bi].grad_dtype, value)
    rep = grads[bi][k]
    if hc.cfg["layout"] == "full":
        rep[w] = enc
        return
    marker = np.zeros(hc.om.buffers[bi].numel, dtype=bool)
    marker[w] = True
    loc = np.nonzero(hc.to_local(bi, marker))[0]
    assert len(loc) == 1, "planted element outside the selected rank's shard"
    rep[loc[0]] = enc


def plant_sites(hc):
    """Buffer positions of the selected ranks' param elements to plant at:
    the first, a middle and the last element of the first, a middle and the
    last piece of each buffer (last elements are often ragged run ends)."""
    sites = []
    for bi in range(len(hc.om.buffers)):
        pieces = [v for r in hc.ranks for _, _, v in hc.om.rank_pieces(bi, r)]
        if not pieces:
            continue
        for v in {id(p): p for p in (pieces[0], pieces[len(pieces) // 2], pieces[-1])}.values():
            g = v["gbuf_world"]
            for w in sorted({g.start, (g.start + g.end) // 2, g.end - 1}):
                sites.append((bi, w))
    return sites


def amax_equal(dev, want):
    """Bit-exact comparison of float32 results with the oracle's (float32, or
    float64 holding float32 values), except that a NaN matches any NaN: IEEE
    754 leaves the payload of a NaN result open, and the GPU returns its
    canonical NaN where the CPU passes an operand's payload on."""
    dev = np.asarray(dev, np.float32)
    want = np.asarray(want, np.float64).astype(np.float32)
    nd, nw = np.isnan(dev), np.isnan(want)
    return bool(np.array_equal(nd, nw) and np.array_equal(dev[~nd].view(np.uint32), want[~nw].view(np.uint32)))


def run_check(cfg, plants_per_step, staged_group=None):
    """Steps a workload with the grad check on both sides.  plants_per_step:
    one list per step of (site index, replica, value) planted at
    plant_sites(hc)[site index]; sites wrap around.  Returns (ok, report)."""
    torch_ = __import__("torch")
    D = dopt()
    hc = HostCase(cfg)
    dc = DeviceCase(hc)
    sites = plant_sites(hc)
    total = D.dopt_total_buckets(hc.pm)
    report, ok = [], True
    streams = [torch_.cuda.Stream() for _ in range(2)]
    for t_step, plants in enumerate(plants_per_step, start=1):
        grads = hc.grads(t_step)
        for site, k, value in plants:
            bi, w = sites[site % len(sites)]
            plant(hc, grads, bi, k % hc.n_rep, w, value)
        t = hc.t_applied + 1
        before = snapshot(hc)
        ores = oracle.step(hc.om, hc.ranks, grads, hc.state, hc.params, cfg["hp"], t,
                           inv_scale=float(np.float32(1.0 / cfg["loss_scale"])),
                           max_norm=cfg["max_norm"], layout=cfg["layout"], n_inst=cfg["n_inst"],
                           average=cfg["average"], check_grads=True)
        amax = dc._alloc(hc.n_rep * total, torch_.float32).view(hc.n_rep, total).fill_(12345.0)
        reps = [[dc._up(r) for r in g] for g in grads]
        if staged_group:
            found, norm = staged_step(dc, reps, t, staged_group, streams, grad_amax=amax)
        else:
            args = dc.step_args(reps, t)
            args.set_grad_check(amax)
            found, norm = D.dopt_step(args)
        good = amax_equal(amax.cpu().numpy(), ores["grad_amax"])
        if not good:
            report.append(f"step {t_step}: grad check table differs:\n{amax.cpu().numpy()}\n"
                          f"oracle:\n{ores['grad_amax']}")
        fused_ws = dc.ws
        if staged_group:
            dc.ws = dc.bws  # the step statistics live in the staged workspace
        good &= compare_step(hc, dc, ores, found, norm, before, report)
        dc.ws = fused_ws
        report.append(f"step {t_step}: found_inf={found} ok={good}")
        ok &= good
        if not ores["found_inf"]:
            hc.t_applied += 1
    return ok, report


def decode_main(raw, gdt, inv_scale, n):
    """The fp32 main grads held in a main-grad buffer after a fused or
    bucket-staged step: for an fp32 grad buffer the buffer itself; for a
    bf16/fp16 grad buffer the first n 16-bit words hold the reduced grads in
    the grad dtype, and main = fp32(word) * inv_scale, one fp32 rounding."""
    raw = np.asarray(raw)
    if gdt == F32:
        return raw[:n]
    bits = raw.view(np.uint16)[:n]
    if gdt == BF16:
        vals = (bits.astype(np.uint32) << 16).view(np.float32)
    else:
        vals = bits.view(np.float16).astype(np.float32)
    return vals * np.float32(inv_scale)


def ulp16(a, b):
    """Distance in ulps between 16-bit float bit patterns (bf16 or fp16)."""
    def key(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7FFF), x)
    return np.abs(key(a) - key(b))


def state_close(got, want, before):
    """fp32 state tolerance: 4 ulp, or 1e-6 relative to the operand scale."""
    got = np.asarray(got, np.float32)
    want = np.asarray(want, np.float32)
    scale = np.maximum(np.maximum(np.abs(before), np.abs(want)), np.float32(1e-30))
    with np.errstate(invalid="ignore"):  # identical non-finite values pass by ulp distance
        return (oracle.float_ulp_diff(got, want) <= 4) | (
            np.abs(got.astype(np.float64) - want.astype(np.float64)) <= 1e-6 * scale)


def compare_step(hc, dc, ores, found, norm, before, report, compact=True, ws=None):
    """Compares the device state after a step with the oracle's.  `before`
    holds the oracle's state before the step; compact: the step was fused or
    bucket-staged, so 16-bit grad buffers left their main grads in compact
    form (decode_main); ws: the workspace that holds the step's statistics
    (the bucket-staged step's own, or by default the fused step's; False:
    the statistics sit where no caller can read them, and are not checked).  Appends
    findings to report and returns True when every check passes."""
    ok = True
    if hasattr(dc, "check_guards") and not dc.check_guards():
        report.append("a write landed outside a device buffer (guard bytes changed)")
        ok = False
    if bool(found) != bool(ores["found_inf"]):
        report.append(f"found_inf device={found} oracle={ores['found_inf']}")
        return False
    if not found:
        rel = abs(norm - ores["norm"]) / max(ores["norm"], 1e-30)
        if not rel <= 1e-5:
            report.append(f"grad_norm device={norm} oracle={ores['norm']} rel={rel:.3g}")
            ok = False
    stats = None if ws is False else dopt().dopt_read_step_stats(dc.ws if ws is None else ws)
    if stats is not None and stats["num_zeros"] != ores["num_zeros"]:
        report.append(f"num_zeros device={stats['num_zeros']} oracle={ores['num_zeros']}")
        ok = False
    params, master, exp_avg, exp_avg_sq, mains = dc.download()
    for bi, buf in enumerate(hc.om.buffers):
        mask = hc.piece_mask(bi)
        st = hc.state[bi]
        om_ = ores["main"][bi]
        got_main = mains[bi]
        if compact:
            got_main = decode_main(got_main, buf.grad_dtype, np.float32(1.0 / hc.cfg["loss_scale"]),
                                   len(st["exp_avg"]))
        if not amax_equal(got_main[mask], om_[mask]):
            report.append(f"buffer {bi}: main grad differs")
            ok = False
        checks = [("exp_avg", exp_avg[bi], st["exp_avg"], before[bi]["exp_avg"]),
                  ("exp_avg_sq", exp_avg_sq[bi], st["exp_avg_sq"], before[bi]["exp_avg_sq"])]
        if "master" in st:
            checks.append(("master", master[bi], st["master"], before[bi]["master"]))
        for name, g, w, b in checks:
            good = state_close(g[mask], w[mask], b[mask])
            if not good.all():
                report.append(f"buffer {bi}: {name} off at {int((~good).sum())} elements, "
                              f"max ulp {int(oracle.float_ulp_diff(g[mask], w[mask]).max())}")
                ok = False
        p_dev, p_or = params[bi], hc.params[bi]
        if buf.param_dtype == F32:
            pm = np.zeros(buf.numel, bool)
            for r in hc.ranks:
                for _, _, v in hc.om.rank_pieces(bi, r):
                    pm[v["gbuf_world"].start:v["gbuf_world"].end] = True
            good = state_close(p_dev[pm], p_or[pm], before[bi]["param"][pm])
            if not good.all():
                report.append(f"buffer {bi}: fp32 param off at {int((~good).sum())} elements")
                ok = False
            if not np.array_equal(p_dev[~pm].view(np.uint32), p_or[~pm].view(np.uint32)):
                report.append(f"buffer {bi}: fp32 param changed outside the shards")
                ok = False
        else:
            d = ulp16(p_dev, p_or)
            if d.max() > 1:
                report.append(f"buffer {bi}: 16-bit param off by {int(d.max())} ulp at "
                              f"{int((d > 1).sum())} elements")
                ok = False
    return ok


def snapshot(hc):
    return [dict({k: v.copy() for k, v in st.items()}, param=p.copy())
            for st, p in zip(hc.state, hc.params)]


def run_parity(cfg, steps=None, separate=False):
    """Steps a workload on both sides and returns (all ok, report lines)."""
    hc = HostCase(cfg)
    dc = DeviceCase(hc)
    report = []
    ok = True
    for t_step in range(1, (steps or cfg["steps"]) + 1):
        grads = hc.grads(t_step)
        t = hc.t_applied + 1
        before = snapshot(hc)
        ores = hc.oracle_step(grads, t)
        found, norm = dc.step_separate(grads, t) if separate else dc.step(grads, t)
        good = compare_step(hc, dc, ores, found, norm, before, report, compact=not separate)
        report.append(f"step {t_step} (t={t}): found_inf={found} norm={norm:.9g} "
                      f"oracle={ores['norm']:.9g} coef={ores['coef']:.9g} ok={good}")
        ok &= good
        if not ores["found_inf"]:
            hc.t_applied += 1
    return ok, report


# ----------------------------------------------------------------------------
# Full-size workloads: inputs filled on the device by the generator, the
# oracle streams the grad norm over every element and recomputes sampled
# elements one by one.

class FullCase:
    """A workload at its full size on the GPU, checked on samples."""

    def __init__(self, cfg):
        import torch
        D = dopt()
        self.torch, self.cfg = torch, cfg
        dp, bs = cfg["dp"], cfg["bucket_size"]
        self.om = oracle.ShardMap(cfg["params"], dp, bs, cfg["grad_reduce_in_fp32"])
        self.pm = D.dopt_build_shard_map(cfg["params"], dp, -1 if bs is None else bs,
                                         cfg["grad_reduce_in_fp32"], False)
        self.all_ranks = cfg["ranks"] == "all"
        self.ranks = list(range(dp)) if self.all_ranks else list(cfg["ranks"])
        self.rank_arg = D.ALL_RANKS if self.all_ranks else self.ranks[0]
        self.n_rep = dp * cfg["n_inst"]
        self.seed = cfg["seed"]
        self.stream = torch.cuda.current_stream().cuda_stream
        dev = torch.device("cuda")
        tdt = {F32: torch.float32, BF16: torch.int16, F16: torch.int16}
        self.pkey = synth.key(self.seed, synth.STREAM_PARAM, 0, 0)
        self.params, self.master, self.m, self.v, self.main, self.reps = [], [], [], [], [], []
        for bi, buf in enumerate(self.om.buffers):
            S = self.om.shard_numel(bi)
            n_local = len(self.ranks) * S
            p = torch.empty(buf.numel, dtype=tdt[buf.param_dtype], device=dev)
            synth.cuda_normal_(p.data_ptr(), buf.numel, self.pkey, 0, cfg["param_sigma"],
                               KIND[buf.param_dtype], self.stream)
            self.params.append(p)
            if buf.param_dtype == F32:
                self.master.append(None)
            else:
                mt = torch.empty(n_local, dtype=torch.float32, device=dev)
                self._fill_local(bi, mt, self.pkey, cfg["param_sigma"], VALUE_KIND[buf.param_dtype])
                self.master.append(mt)
            self.m.append(torch.zeros(n_local, dtype=torch.float32, device=dev))
            self.v.append(torch.zeros(n_local, dtype=torch.float32, device=dev))
            self.main.append(torch.zeros(n_local, dtype=torch.float32, device=dev))
            n_rep_elems = buf.numel if cfg["layout"] == "full" else S
            self.reps.append([torch.empty(n_rep_elems, dtype=tdt[buf.grad_dtype], device=dev)
                              for _ in range(self.n_rep)])
        self.ws_bytes = D.dopt_workspace_bytes(self.pm, self.rank_arg)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()

    def _fill_local(self, bi, t, key, sigma, kind):
        S = self.om.shard_numel(bi)
        for slot, r in enumerate(self.ranks):
            for b in range(len(self.om.buffers[bi].buckets)):
                rg = self.om.bucket_world_range(bi, b, r)
                off = slot * S + self.om.bucket_shard_base(bi, b)
                synth.cuda_normal_(t.data_ptr() + off * t.element_size(), rg.size, key, rg.start,
                                   sigma, kind, self.stream)

    def fill_grads(self, t):
        cfg = self.cfg
        for bi, buf in enumerate(self.om.buffers):
            for k, rep in enumerate(self.reps[bi]):
                key = synth.key(self.seed, synth.STREAM_GRAD, t, k)
                if cfg["layout"] == "full":
                    synth.cuda_normal_(rep.data_ptr(), buf.numel, key, 0, cfg["grad_sigma"],
                                       KIND[buf.grad_dtype], self.stream)
                else:
                    self._fill_local(bi, rep, key, cfg["grad_sigma"], KIND[buf.grad_dtype])
        self.torch.cuda.synchronize()

    def step(self, t, grad_amax=None):
        D = dopt()
        cfg = self.cfg
        args = D.StepArgs(self.pm, self.rank_arg, self.reps, self.main, self.master, self.m, self.v,
                          self.params, cfg["hp"], t, self.ws, self.ws_bytes,
                          n_instances=cfg["n_inst"],
                          layout=D.LAYOUT_FULL_BUFFER if cfg["layout"] == "full" else D.LAYOUT_SHARD_ONLY,
                          average_in_collective=cfg["average"],
                          inv_loss_scale=float(np.float32(1.0 / cfg["loss_scale"])),
                          max_norm=cfg["max_norm"], stream=self.torch.cuda.current_stream())
        if grad_amax is not None:
            args.set_grad_check(grad_amax)
        return D.dopt_step(args)

    def pieces(self):
        """(buffer, slot, param id, flat offset, buffer offset, length) of
        every param piece of the selected ranks."""
        out = []
        for bi in range(len(self.om.buffers)):
            S = self.om.shard_numel(bi)
            for slot, r in enumerate(self.ranks):
                for pid, _, v in self.om.rank_pieces(bi, r):
                    out.append((bi, slot, pid, slot * S + v["shard_offset"], v["gbuf_world"].start,
                                v["gbuf_local"].size))
        return out

    def oracle_sumsq(self, t, chunk=1 << 22):
        """The oracle's fp64 sum of squares of every main grad of step t,
        streamed from the generator, in parallel over chunks of the pieces
        (threads: the C oracle releases the GIL)."""
        import os
        from concurrent.futures import ThreadPoolExecutor
        cfg = self.cfg
        keys = [synth.key(self.seed, synth.STREAM_GRAD, t, k) for k in range(self.n_rep)]
        inv = float(np.float32(1.0 / cfg["loss_scale"]))
        jobs = []
        for bi, slot, pid, lo, w, n in self.pieces():
            gdt = self.om.buffers[bi].grad_dtype
            for o in range(0, n, chunk):
                jobs.append((gdt, w + o, min(chunk, n - o)))
        fac = synth.factor(cfg["grad_sigma"])

        def run(j):
            return oracle.stream_sumsq(keys, j[0], fac, j[1], j[2], inv, cfg["n_inst"], cfg["average"])
        with ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
            res = list(ex.map(run, jobs))
        return sum(r[0] for r in res), sum(r[1] for r in res)

    def choose_samples(self, n_random, seed=0):
        """First and last element of every piece plus random elements."""
        rng = np.random.RandomState(seed)
        pcs = self.pieces()
        out = []
        for bi, slot, pid, lo, w, n in pcs:
            out.append((bi, pid, lo, w))
            out.append((bi, pid, lo + n - 1, w + n - 1))
            for cut in range(1 << 30, n, 1 << 30):  # both sides of a 2^30-element run cut
                out.append((bi, pid, lo + cut - 1, w + cut - 1))
                out.append((bi, pid, lo + cut, w + cut))
        lens = np.array([p[5] for p in pcs], dtype=np.float64)
        pick = rng.choice(len(pcs), size=n_random, p=lens / lens.sum())
        for i in pick:
            bi, slot, pid, lo, w, n = pcs[i]
            o = int(rng.randint(0, n))
            out.append((bi, pid, lo + o, w + o))
        return sorted(set(out))

    def initial_sample_state(self, samples):
        cfg = self.cfg
        st = {}
        for bi in range(len(self.om.buffers)):
            sel = [s for s in samples if s[0] == bi]
            if not sel:
                continue
            w = np.array([s[3] for s in sel], dtype=np.uint64)
            pdt = self.om.buffers[bi].param_dtype
            kind = synth.OUT_F32 if pdt == F32 else VALUE_KIND[pdt]
            st[bi] = {"sel": sel, "master": synth.normal_at(w, self.pkey, cfg["param_sigma"], kind),
                      "exp_avg": np.zeros(len(sel), np.float32),
                      "exp_avg_sq": np.zeros(len(sel), np.float32)}
        return st

    def oracle_samples(self, st, t_step, t, coef, clip):
        """Advances the sampled elements' state by one applied step (oracle).
        Returns the main grads per buffer; st is updated in place and gains
        the expected 16-bit param bits under "param"."""
        cfg = self.cfg
        L = oracle.lib()
        h = oracle.Hparams(**cfg["hp"])
        mains = {}
        for bi, s in st.items():
            buf = self.om.buffers[bi]
            w = np.array([x[3] for x in s["sel"]], dtype=np.uint64)
            reps = [synth.normal_at(w, synth.key(self.seed, synth.STREAM_GRAD, t_step, k),
                                    cfg["grad_sigma"], KIND[buf.grad_dtype])
                    for k in range(self.n_rep)]
            main, _ = oracle.reduce_prepare(reps, buf.grad_dtype, 0, len(w),
                                            float(np.float32(1.0 / cfg["loss_scale"])),
                                            cfg["n_inst"], cfg["average"])
            mains[bi] = main
            if t is None:
                continue
            wd = np.array([float(cfg["params"][x[1]].get("wd_mult", 1.0)) for x in s["sel"]])
            out = np.zeros(len(w), np.uint16 if buf.param_dtype != F32 else np.float32)
            for val in np.unique(wd):
                idx = np.nonzero(wd == val)[0]
                sub = {k: np.ascontiguousarray(s[k][idx]) for k in ("master", "exp_avg", "exp_avg_sq")}
                sub_main = np.ascontiguousarray(main[idx])
                sub_out = np.zeros(len(idx), out.dtype)
                L.or_adamw_run(sub_main.ctypes.data, len(idx), coef, int(clip), sub["master"].ctypes.data,
                               sub["exp_avg"].ctypes.data, sub["exp_avg_sq"].ctypes.data,
                               oracle.ctypes_byref(h), float(val), t,
                               sub_out.ctypes.data if buf.param_dtype != F32 else None,
                               buf.param_dtype)
                for k in sub:
                    s[k][idx] = sub[k]
                out[idx] = sub_out if buf.param_dtype != F32 else sub["master"]
            s["param"] = out
        return mains

    def device_samples(self, st):
        torch = self.torch
        got = {}
        for bi, s in st.items():
            lo = torch.tensor([x[2] for x in s["sel"]], dtype=torch.int64, device="cuda")
            w = torch.tensor([x[3] for x in s["sel"]], dtype=torch.int64, device="cuda")
            buf = self.om.buffers[bi]
            if buf.grad_dtype == F32:
                main = self.main[bi][lo].cpu().numpy()
            else:  # compact main grads (decode_main)
                main = decode_main(self.main[bi].view(torch.int16)[lo].cpu().numpy(), buf.grad_dtype,
                                   np.float32(1.0 / self.cfg["loss_scale"]), len(s["sel"]))
            g = {"main": main, "exp_avg": self.m[bi][lo].cpu().numpy(),
                 "exp_avg_sq": self.v[bi][lo].cpu().numpy()}
            p = self.params[bi][w].cpu().numpy()
            g["param"] = p.view(np.uint16) if p.dtype == np.int16 else p
            g["master"] = (self.master[bi][lo].cpu().numpy() if self.master[bi] is not None
                           else g["param"])
            got[bi] = g
        return got

    # ---- element-wise parity on a window of whole buckets ------------------

    def window_buckets(self, min_elems=64 << 20):
        """Whole buckets to compare element by element: every bucket of every
        buffer after the first (the small fp32 norm-weight buffers), and of
        buffer 0 its first, middle and last bucket, then more buckets taken
        alternately from the front and the back until the window holds at
        least min_elems of the selected ranks' buffer elements (or all of
        them).  Returns sorted (buffer, bucket) pairs."""
        om = self.om
        per = len(self.ranks)
        out = set()
        size = 0

        def take(bi, b):
            nonlocal size
            if (bi, b) not in out:
                out.add((bi, b))
                size += per * (om.buffers[bi].buckets[b].numel // om.dp)

        for bi in range(1, len(om.buffers)):
            for b in range(len(om.buffers[bi].buckets)):
                take(bi, b)
        nbk = len(om.buffers[0].buckets)
        for b in (0, nbk // 2, nbk - 1):
            take(0, b)
        lo, hi = 1, nbk - 2
        while size < min_elems and lo <= hi:
            take(0, lo)
            if size < min_elems:
                take(0, hi)
            lo, hi = lo + 1, hi - 1
        return sorted(out)

    def window_pieces(self, buckets):
        """Param pieces of the selected ranks inside the given buckets, per
        buffer: {bi: [(param id, flat-shard offset, buffer offset, length,
        offset in the window arrays)]}."""
        sel = {}
        for bi, b in buckets:
            sel.setdefault(bi, set()).add(b)
        out = {}
        for bi, bs in sorted(sel.items()):
            S = self.om.shard_numel(bi)
            lst, off = [], 0
            for slot, r in enumerate(self.ranks):
                for pid, b, v in self.om.rank_pieces(bi, r):
                    if b in bs:
                        n = v["gbuf_local"].size
                        lst.append((pid, slot * S + v["shard_offset"], v["gbuf_world"].start, n, off))
                        off += n
            out[bi] = lst
        return out

    def window_initial_state(self, pieces):
        """The oracle's starting state of the window (master from the
        generator, m = v = 0), per buffer: float32 arrays master, exp_avg,
        exp_avg_sq (for an fp32 buffer the master is the param itself)."""
        cfg = self.cfg
        st = {}
        for bi, lst in pieces.items():
            n = lst[-1][4] + lst[-1][3] if lst else 0
            pdt = self.om.buffers[bi].param_dtype
            kind = synth.OUT_F32 if pdt == F32 else VALUE_KIND[pdt]
            master = np.empty(n, np.float32)
            for pid, lo, w, k, off in lst:
                master[off:off + k] = synth.normal(k, self.pkey, w, cfg["param_sigma"], kind)
            st[bi] = {"master": master, "exp_avg": np.zeros(n, np.float32),
                      "exp_avg_sq": np.zeros(n, np.float32)}
        return st

    def window_device(self, pieces):
        """The device's window: per buffer main (fp32, decoded from the
        compact form for 16-bit grads), master, exp_avg, exp_avg_sq and param
        (16-bit bits, or fp32) arrays in window order."""
        torch = self.torch
        inv = np.float32(1.0 / self.cfg["loss_scale"])
        got = {}
        for bi, lst in pieces.items():
            buf = self.om.buffers[bi]
            n = lst[-1][4] + lst[-1][3] if lst else 0
            g = {k: np.empty(n, np.float32) for k in ("main", "master", "exp_avg", "exp_avg_sq")}
            g["param"] = np.empty(n, np.uint16 if buf.param_dtype != F32 else np.float32)
            for pid, lo, w, k, off in lst:
                if buf.grad_dtype == F32:
                    g["main"][off:off + k] = self.main[bi][lo:lo + k].cpu().numpy()
                else:
                    raw = self.main[bi].view(torch.int16)[lo:lo + k].cpu().numpy()
                    g["main"][off:off + k] = decode_main(raw, buf.grad_dtype, inv, k)
                g["exp_avg"][off:off + k] = self.m[bi][lo:lo + k].cpu().numpy()
                g["exp_avg_sq"][off:off + k] = self.v[bi][lo:lo + k].cpu().numpy()
                p = self.params[bi][w:w + k].cpu().numpy()
                g["param"][off:off + k] = p.view(np.uint16) if p.dtype == np.int16 else p
                if self.master[bi] is not None:
                    g["master"][off:off + k] = self.master[bi][lo:lo + k].cpu().numpy()
                else:
                    g["master"][off:off + k] = g["param"][off:off + k]
            got[bi] = g
        return got

    def window_oracle_step(self, pieces, st, t_step, t, coef, clip, chunk=1 << 20):
        """Advances the window's oracle state by one applied step (t None:
        only the main grads).  The main grads of every element are redrawn
        from the generator (oracle.stream_reduce_prepare); AdamW and the
        write-back run per param piece (or_adamw_run), in chunks on a thread
        pool (the C oracle releases the GIL).  Returns per buffer the main
        grads and the expected params (16-bit bits, or fp32)."""
        import os
        from concurrent.futures import ThreadPoolExecutor
        cfg = self.cfg
        L = oracle.lib()
        h = oracle.Hparams(**cfg["hp"])
        keys = [synth.key(self.seed, synth.STREAM_GRAD, t_step, k) for k in range(self.n_rep)]
        fac = synth.factor(cfg["grad_sigma"])
        inv = float(np.float32(1.0 / cfg["loss_scale"]))
        res, jobs = {}, []
        for bi, lst in pieces.items():
            buf = self.om.buffers[bi]
            n = st[bi]["master"].size
            main = np.empty(n, np.float32)
            param = np.empty(n, np.uint16) if buf.param_dtype != F32 else st[bi]["master"]
            res[bi] = {"main": main, "param": param}
            for pid, lo, w, k, off in lst:
                wd = float(cfg["params"][pid].get("wd_mult", 1.0))
                for o in range(0, k, chunk):
                    jobs.append((bi, w + o, off + o, min(chunk, k - o), wd))

        def run(j):
            bi, w, a, k, wd = j
            buf = self.om.buffers[bi]
            main = res[bi]["main"][a:a + k]
            _, bad = oracle.stream_reduce_prepare(keys, buf.grad_dtype, fac, w, k, out=main,
                                                  inv_scale=inv, n_inst=cfg["n_inst"],
                                                  average=cfg["average"])
            if t is None:
                return bad
            s = st[bi]
            out = None if buf.param_dtype == F32 else res[bi]["param"][a:a + k].ctypes.data
            L.or_adamw_run(main.ctypes.data, k, coef, int(clip), s["master"][a:a + k].ctypes.data,
                           s["exp_avg"][a:a + k].ctypes.data, s["exp_avg_sq"][a:a + k].ctypes.data,
                           oracle.ctypes_byref(h), wd, t, out, buf.param_dtype)
            return bad
        with ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
            bad = sum(ex.map(run, jobs))
        return res, bad


def window_compare(got, want, prev, chunk=1 << 22):
    """Element-wise parity of a window, in chunks: main grads bit-exact,
    master / m / v within the state tolerance, 16-bit params within 1 ulp,
    fp32 params (the master itself) within the state tolerance.  Elements
    whose bits are equal pass at once; only the others are measured against
    the tolerance.  Returns a list of findings (empty when every element
    passes)."""
    bad = []
    for bi in got:
        g, w, p = got[bi], want[bi], prev[bi]
        n = g["main"].size
        for a in range(0, n, chunk):
            b = min(n, a + chunk)
            gm, wm = g["main"][a:b], w["main"][a:b]
            if not (np.array_equal(gm.view(np.uint32), wm.view(np.uint32)) or amax_equal(gm, wm)):
                bad.append(f"buffer {bi}: main grad differs in [{a}, {b})")
            for k in ("master", "exp_avg", "exp_avg_sq"):
                gk, wk = g[k][a:b], w[k][a:b]
                diff = np.nonzero(gk.view(np.uint32) != wk.view(np.uint32))[0]
                if diff.size:
                    ok = state_close(gk[diff], wk[diff], p[k][a:b][diff])
                    if not ok.all():
                        bad.append(f"buffer {bi}: {k} off at {int((~ok).sum())} elements in [{a}, {b})")
            if g["param"].dtype == np.uint16:
                gp, wp = g["param"][a:b], w["param"][a:b]
                diff = np.nonzero(gp != wp)[0]
                if diff.size:
                    d = ulp16(gp[diff], wp[diff])
                    if d.max() > 1:
                        bad.append(f"buffer {bi}: param off by {int(d.max())} ulp in [{a}, {b})")
    return bad


def window_chunks(pieces, state, max_elems):
    """Splits a window into consecutive groups of whole param pieces of at
    most max_elems elements (a piece longer than that is a group of its own):
    yields (sub-pieces with offsets from the group's start, views of the
    window state arrays over the group)."""
    for bi, lst in pieces.items():
        i = 0
        while i < len(lst):
            j, size = i, 0
            while j < len(lst) and (j == i or size + lst[j][3] <= max_elems):
                size += lst[j][3]
                j += 1
            base = lst[i][4]
            sub = {bi: [(pid, lo, w, k, off - base) for pid, lo, w, k, off in lst[i:j]]}
            views = {bi: {key: arr[base:base + size] for key, arr in state[bi].items()}}
            yield sub, views
            i = j
