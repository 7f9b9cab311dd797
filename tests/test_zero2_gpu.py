"""The ZeRO-2 step flow: grads streamed bucket by bucket through two staging
buffers per replica (DOPT_LAYOUT_BUCKET), so a rank never holds more than two
buckets of full grads; each bucket is reduced into the rank's grad shard as
soon as its grads are in, and its staging buffer is refilled with a later
bucket's grads once that reduce has run.  DeepSpeed page, ZeRO stage 2 step
(reduce-scatter, update the rank's partition, all-gather); ZeRO ledger
page, section 2 (2P + 14P/N per card).

Every step is compared with the oracle's step on the whole grad buffers,
through a skipped step, and the rank's device memory for a 16-bit model is
checked against dopt_memory_ledger(P, N, 2): params 2P, grad shard 2P/N
(the main grads between the passes, kept in the grad dtype) and fp32
master, m, v 12P/N -- besides the staging ring (two buckets per emulated
replica, standing in for the grads in flight in the collective) and the
workspace."""

import numpy as np
import pytest

from synth import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gpu_harness as H  # noqa: E402

TORCH_DT = {H.F32: torch.float32, H.BF16: torch.int16, H.F16: torch.int16}


class Zero2Rank:
    """One device case stepped by streaming its replica grads through a
    two-slot staging ring per replica and buffer."""

    def __init__(self, hc):
        D = H.dopt()
        self.hc = hc
        self.dc = H.DeviceCase(hc)
        om = hc.om
        self.ws_bytes = D.dopt_workspace_bytes_bucketed(hc.pm, hc.rank_arg)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device="cuda")
        self.slots = []  # [buffer][slot][replica] device tensors of the buffer's largest bucket
        for buf in om.buffers:
            n = max(b.numel for b in buf.buckets)
            self.slots.append([[torch.empty(n, dtype=TORCH_DT[buf.grad_dtype], device="cuda")
                                for _ in range(hc.n_rep)] for _ in range(2)])
        self.producer = torch.cuda.Stream()
        self.reducer = torch.cuda.Stream()

    def staging_bytes(self):
        return sum(t.numel() * t.element_size() for s in self.slots for ring in s for t in ring)

    def step(self, grads, t, grad_amax=None):
        """grads: the oracle's whole-buffer replica arrays; grad_amax: a
        device table for the pre-reduction grad check, or None.  Returns
        (found_inf, norm) of the step."""
        D = H.dopt()
        hc, dc = self.hc, self.dc
        host = [[torch.from_numpy(r.view(np.int16) if r.dtype == np.uint16 else r).pin_memory()
                 for r in reps] for reps in grads]
        args = dc.step_args([ring for ring in (s[0] for s in self.slots)], t)
        args.c.layout = D.LAYOUT_BUCKET
        if grad_amax is not None:
            args.set_grad_check(grad_amax)
        args.c.workspace, args.c.workspace_bytes = self.ws.data_ptr(), self.ws_bytes
        main = torch.cuda.current_stream()
        self.producer.wait_stream(main)
        self.reducer.wait_stream(main)
        consumed = [[None, None] for _ in self.slots]
        n_stream = 0
        for bi, buf in enumerate(hc.om.buffers):
            for k, bk in enumerate(buf.buckets):  # bucket 0 first: its grads are ready first
                slot = n_stream % 2
                n_stream += 1
                ring = self.slots[bi][slot]
                if consumed[bi][slot] is not None:  # the reduce that read this slot has run
                    self.producer.wait_event(consumed[bi][slot])
                with torch.cuda.stream(self.producer):
                    for r in range(hc.n_rep):
                        ring[r][:bk.numel].copy_(host[bi][r][bk.offset:bk.offset + bk.numel],
                                                 non_blocking=True)
                    ready = torch.cuda.Event()
                    ready.record(self.producer)
                self.reducer.wait_event(ready)
                args.set_replicas(bi, ring)
                args.set_stream(self.reducer)
                D.dopt_step_reduce_buckets(args, bi, k, 1)
                done = torch.cuda.Event()
                done.record(self.reducer)
                consumed[bi][slot] = done
        main.wait_stream(self.reducer)
        args.set_stream(main)
        d_found = torch.zeros(1, dtype=torch.int32, device="cuda")
        d_norm = torch.zeros(1, dtype=torch.float32, device="cuda")
        D.dopt_step_finalize(args, d_found, d_norm)
        for bi, buf in enumerate(hc.om.buffers):
            for k in reversed(range(len(buf.buckets))):
                D.dopt_step_update_buckets(args, bi, k, 1)
        torch.cuda.synchronize()
        return bool(d_found.item()), float(d_norm.item())


def _cfg(workload, **kw):
    cfg = dict(W.mini(workload), layout="full")  # the oracle reads whole buffers
    cfg.update(kw)
    return cfg


@pytest.mark.parametrize("cfg", [
    _cfg("llama_7b_dp8_rank0"),
    _cfg("llama_7b_dp8_rank0", grad_reduce_in_fp32=False, name="llama_bf16_grads"),
    _cfg("gpt2_small_dp8"),  # all ranks; an inf at step 2 skips the step
    _cfg("llama_1p3b_fp16_dp8"),
    _cfg("llama_7b_dp16_2x8_1m"),
], ids=lambda c: c["name"])
def test_zero2_streaming_matches_oracle(cfg):
    hc = H.HostCase(cfg)
    rank = Zero2Rank(hc)
    assert all(len(b.buckets) >= 2 for b in hc.om.buffers[:1])  # the ring is reused
    report, found_seq = [], []
    for step in (1, 2, 3):
        grads = hc.grads(step)
        t = hc.t_applied + 1
        before = H.snapshot(hc)
        ores = hc.oracle_step(grads, t)
        found, norm = rank.step(grads, t)
        ok = H.compare_step(hc, rank.dc, ores, found, norm, before, report, ws=rank.ws)
        assert ok, "\n".join(report)
        found_seq.append(found)
        if not found:
            hc.t_applied += 1
    assert found_seq == [False, cfg.get("inf_at") is not None, False]


@pytest.mark.parametrize("dp", [4, 8])
def test_zero2_rank_memory_equals_the_ledger(dp):
    """A bf16 model with bf16 grads: what the rank holds for the step -- the
    whole param buffer, the 16-bit main grads of its shard and the fp32
    master, m and v of its shard -- is dopt_memory_ledger(P, N, 2); the
    staging ring (two buckets per emulated replica) and the workspace come on
    top.  The steps themselves allocate no device memory, and they match the
    oracle with the main grads given only 2 bytes per shard element."""
    D = H.dopt()
    params = [dict(name=f"w{i}", numel=n, dtype=W.BF16)
              for i, n in enumerate((300_000, 65_536, 1_000_000, 4_096, 700_000))]
    cfg = W._cfg(name="zero2_ledger", params=params, dp=dp, bucket_size=400_000,
                 grad_reduce_in_fp32=False, layout="full", ranks=[1], steps=3, seed=41)
    hc = H.HostCase(cfg)
    assert len(hc.om.buffers) == 1 and len(hc.om.buffers[0].buckets) >= 3
    P = hc.om.buffers[0].numel
    S = P // dp
    rank = Zero2Rank(hc)
    dc = rank.dc
    # the rank's main grads sized as the staged step uses them for 16-bit
    # grads: 2 bytes per shard element (an fp32 view of half as many)
    main16 = dc._alloc(S, torch.int16).zero_()
    dc.main = [main16.view(torch.float32)]
    held = (dc.params[0].numel() * 2 + main16.numel() * 2 +
            sum(t.numel() * 4 for t in (dc.master[0], dc.exp_avg[0], dc.exp_avg_sq[0])))
    assert held == D.dopt_memory_ledger(P, dp, 2)[0] == 2 * P + 14 * (P // dp)
    assert rank.staging_bytes() == 2 * dp * max(b.numel for b in hc.om.buffers[0].buckets) * 2
    report = []
    free = []
    for step in (1, 2, 3):
        grads = hc.grads(step)
        before = H.snapshot(hc)
        ores = hc.oracle_step(grads, step)
        found, norm = rank.step(grads, step)
        assert H.compare_step(hc, dc, ores, found, norm, before, report, ws=rank.ws), "\n".join(report)
        hc.t_applied += 1
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
    assert free[1] == free[2]  # after the first step (pinned copies, events) nothing more is held


@pytest.mark.parametrize("name", ["llama_7b_dp8_rank0", "gpt2_small_dp8"])
def test_zero2_streaming_grad_check(name):
    """The pre-reduction grad check through the ZeRO-2 flow: each bucket's
    staging buffers are checked as they are reduced, and the table (largest
    |g| per replica and bucket among the elements the step reads) equals
    the oracle's for whole buffers, with a large value and a NaN planted."""
    cfg = dict(_cfg(name), inf_at=None)
    hc = H.HostCase(cfg)
    rank = Zero2Rank(hc)
    D = H.dopt()
    total = D.dopt_total_buckets(hc.pm)
    sites = H.plant_sites(hc)
    report = []
    for step, plants in ((1, [(0, 1, 1.0e3)]), (2, [(len(sites) // 2, hc.n_rep - 1, float("nan"))])):
        grads = hc.grads(step)
        for site, k, value in plants:
            bi, w = sites[site]
            H.plant(hc, grads, bi, k, w, value)
        t = hc.t_applied + 1
        before = H.snapshot(hc)
        ores = H.oracle.step(hc.om, hc.ranks, grads, hc.state, hc.params, cfg["hp"], t,
                             inv_scale=float(np.float32(1.0 / cfg["loss_scale"])), max_norm=cfg["max_norm"],
                             layout="full", n_inst=cfg["n_inst"], average=cfg["average"], check_grads=True)
        amax = torch.full((hc.n_rep, total), 12345.0, dtype=torch.float32, device="cuda")
        found, norm = rank.step(grads, t, grad_amax=amax)
        assert H.amax_equal(amax.cpu().numpy(), ores["grad_amax"]), (step, amax.cpu().numpy(), ores["grad_amax"])
        assert H.compare_step(hc, rank.dc, ores, found, norm, before, report, ws=rank.ws), "\n".join(report)
        assert found == (step == 2)
        if not found:
            hc.t_applied += 1
