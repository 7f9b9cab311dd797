"""Two ranks of one DP=2 optimizer instance, each stepping its own shard
through the bucket-staged entry points and combining their norm statistics
on the device: dopt_step_local_stats writes each rank's sum of squares and
non-finite flag, a device add / max stands in for the all-reduce, and
dopt_step_finalize reads the results through d_global_sumsq /
d_global_found_inf.  Checked against the same composition through host
remote terms (bit for bit) and against the all-ranks oracle step; an inf in
one rank's grads must skip both ranks.  The ranks run one after the other on
one GPU: nothing waits on another launch."""

import numpy as np
import pytest

from synth import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gpu_harness as H  # noqa: E402

CFG = W._cfg(name="two_ranks", params=W.llama(2, 128, 344, 999), dp=2, bucket_size=60_000,
             layout="shard", steps=3, seed=23, grad_sigma=1e-2,
             inf_at=dict(step=2, replica=1, buffer_frac=0.4))


class Rank:
    """One rank's device state and its bucket-staged step arguments."""

    def __init__(self, r):
        self.hc = H.HostCase(dict(CFG, ranks=[r], inf_at=None))
        self.dc = H.DeviceCase(self.hc)
        D = H.dopt()
        self.ws_bytes = D.dopt_workspace_bytes_bucketed(self.hc.pm, r)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device="cuda")
        self.local = torch.zeros(1, dtype=torch.float64, device="cuda")
        self.flag = torch.zeros(1, dtype=torch.int32, device="cuda")

    def reduce(self, grads, t):
        D = H.dopt()
        self.args = self.dc.step_args([[self.dc._up(g) for g in reps] for reps in grads], t)
        self.args.c.workspace, self.args.c.workspace_bytes = self.ws.data_ptr(), self.ws_bytes
        for bi, buf in enumerate(self.hc.om.buffers):
            D.dopt_step_reduce_buckets(self.args, bi, 0, len(buf.buckets))
        D.dopt_step_local_stats(self.args, self.local, self.flag)

    def finish(self):
        D = H.dopt()
        d_found = torch.zeros(1, dtype=torch.int32, device="cuda")
        d_norm = torch.zeros(1, dtype=torch.float32, device="cuda")
        D.dopt_step_finalize(self.args, d_found, d_norm)
        for bi, buf in enumerate(self.hc.om.buffers):
            for k in reversed(range(len(buf.buckets))):
                D.dopt_step_update_buckets(self.args, bi, k, 1)
        torch.cuda.synchronize()
        return bool(d_found.item()), float(d_norm.item())


def _shard(hc_all, bi, g, r):
    """Rank r's flat shard of a whole-buffer array g of buffer bi."""
    om = hc_all.om
    return np.concatenate([g[om.bucket_world_range(bi, b, r).start:om.bucket_world_range(bi, b, r).end]
                           for b in range(len(om.buffers[bi].buckets))])


def test_two_ranks_combine_statistics_on_the_device():
    hc_all = H.HostCase(dict(CFG, ranks="all", layout="full"))
    dev = [Rank(0), Rank(1)]    # statistics combined on the device
    host = [Rank(0), Rank(1)]   # the same through host remote terms
    t_applied = 0
    for t_step in range(1, CFG["steps"] + 1):
        t = t_applied + 1
        full = hc_all.grads(t_step)  # every rank's grads, with the planted inf of step 2
        before = H.snapshot(hc_all)
        ores = hc_all.oracle_step(full, t)
        for r in (0, 1):
            g = [[_shard(hc_all, bi, x, r) for x in reps] for bi, reps in enumerate(full)]
            dev[r].reduce(g, t)
            host[r].reduce(g, t)
        torch.cuda.synchronize()
        # each rank's local fp64 sum, the same on both paths; together the oracle's
        loc = [float(rk.local.item()) for rk in dev]
        assert loc == [float(rk.local.item()) for rk in host]
        if not ores["found_inf"]:
            assert abs(sum(loc) - ores["sumsq"]) <= 1e-12 * ores["sumsq"]
        dev_before = [rk.dc.download() for rk in dev]
        glob = dev[0].local + dev[1].local
        gflag = torch.maximum(dev[0].flag, dev[1].flag)
        results = []
        for rk in dev:
            rk.args.set_global_stats(glob, gflag)
            results.append(rk.finish())
        for r, rk in enumerate(host):
            other = host[1 - r]
            rk.args.c.remote_sumsq = float(other.local.item())
            rk.args.c.remote_found_inf = int(other.flag.item())
            fh, nh = rk.finish()
            fd, nd = results[r]
            assert (fh, np.float32(nh).tobytes()) == (fd, np.float32(nd).tobytes())
            for a, b in zip(rk.dc.download(), dev[r].dc.download()):
                for x, y in zip(a, b):
                    assert (x is None and y is None) or x.tobytes() == y.tobytes()
        assert all(f == ores["found_inf"] for f, _ in results)
        if ores["found_inf"]:  # skipped on both ranks: nothing moved
            for r, rk in enumerate(dev):
                for a, b in zip(dev_before[r][:4], rk.dc.download()[:4]):
                    for x, y in zip(a, b):
                        assert (x is None and y is None) or x.tobytes() == y.tobytes()
            continue
        for _, n in results:
            assert abs(n - ores["norm"]) <= 1e-5 * ores["norm"]
        for r, rk in enumerate(dev):
            _, master, exp_avg, exp_avg_sq, _ = rk.dc.download()
            for bi in range(len(hc_all.om.buffers)):
                S = hc_all.om.shard_numel(bi)
                sl = slice(r * S, (r + 1) * S)
                mask = hc_all.piece_mask(bi)[sl]
                st = hc_all.state[bi]
                for name, got in (("exp_avg", exp_avg[bi]), ("exp_avg_sq", exp_avg_sq[bi]), ("master", master[bi])):
                    if got is None:
                        continue
                    ok = H.state_close(got[mask], st[name][sl][mask], before[bi][name][sl][mask])
                    assert ok.all(), (t_step, r, bi, name)
        t_applied += 1
    assert t_applied == CFG["steps"] - 1


def test_two_rank_step_captured_in_one_graph():
    """The whole two-rank step -- both ranks' reduces, local statistics, the
    device add and max standing in for the all-reduce, both finalizes and
    updates -- captured in one CUDA graph with device step counters, and
    replayed with fresh grads each step (one of them with an inf): bit for
    bit the eager composition's state."""
    D = H.dopt()
    hc_all = H.HostCase(dict(CFG, ranks="all", layout="full"))

    def shards(t_step):
        full = hc_all.grads(t_step)
        return [[[_shard(hc_all, bi, x, r) for x in reps] for bi, reps in enumerate(full)] for r in (0, 1)]

    def body(ranks, glob, gflag):
        for rk in ranks:
            for bi, buf in enumerate(rk.hc.om.buffers):
                D.dopt_step_reduce_buckets(rk.args, bi, 0, len(buf.buckets))
            D.dopt_step_local_stats(rk.args, rk.local, rk.flag)
        torch.add(ranks[0].local, ranks[1].local, out=glob)
        torch.maximum(ranks[0].flag, ranks[1].flag, out=gflag)
        for rk in ranks:
            D.dopt_step_finalize(rk.args)
            for bi, buf in enumerate(rk.hc.om.buffers):
                for k in reversed(range(len(buf.buckets))):
                    D.dopt_step_update_buckets(rk.args, bi, k, 1)

    def setup(ranks, grads, stream):
        glob = torch.zeros(1, dtype=torch.float64, device="cuda")
        gflag = torch.zeros(1, dtype=torch.int32, device="cuda")
        for rk, g in zip(ranks, grads):
            rk.reps = [[rk.dc._up(x) for x in reps] for reps in g]
            rk.args = rk.dc.step_args(rk.reps, 1, stream=stream)
            rk.args.c.workspace, rk.args.c.workspace_bytes = rk.ws.data_ptr(), rk.ws_bytes
            rk.d_step = torch.zeros(1, dtype=torch.int64, device="cuda")
            rk.args.set_device_step(rk.d_step)
            rk.args.set_global_stats(glob, gflag)
        return glob, gflag

    first = shards(1)
    warm = [Rank(0), Rank(1)]  # runs every kernel once outside the capture
    body(warm, *setup(warm, first, torch.cuda.current_stream()))
    torch.cuda.synchronize()

    graphed = [Rank(0), Rank(1)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        glob, gflag = setup(graphed, first, s)
        with torch.cuda.graph(graph, stream=s):
            body(graphed, glob, gflag)
    torch.cuda.synchronize()

    eager = [Rank(0), Rank(1)]
    t_applied = 0
    for t_step in range(1, CFG["steps"] + 1):
        g = shards(t_step)
        for rk, gr in zip(graphed, g):
            for dst_b, src_b in zip(rk.reps, gr):
                for dst, src in zip(dst_b, src_b):
                    dst.copy_(rk.dc._up(src))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        t = t_applied + 1
        for rk, gr in zip(eager, g):
            rk.reduce(gr, t)
        eg = eager[0].local + eager[1].local
        ef = torch.maximum(eager[0].flag, eager[1].flag)
        found = []
        for rk in eager:
            rk.args.set_global_stats(eg, ef)
            found.append(rk.finish()[0])
        assert found[0] == found[1] == (t_step == 2)
        if not found[0]:
            t_applied += 1
        for a, b in zip(graphed, eager):
            assert int(a.d_step.item()) == t_applied
            for x_arr, y_arr in zip(a.dc.download()[:4], b.dc.download()[:4]):
                for x, y in zip(x_arr, y_arr):
                    assert (x is None and y is None) or x.tobytes() == y.tobytes(), t_step


@pytest.mark.parametrize("seed", range(6))
def test_random_maps_every_rank_on_the_device(seed):
    """Seeded random maps (dtypes, bucket sizes, padding, instances,
    averaging, loss scales) at DP 2 to 4, every rank stepped on its own shard
    with the norm statistics combined on the device, against the all-ranks
    oracle step."""
    import random as _random
    import test_random_gpu as R
    cfg = R._random_cfg(100 + seed)
    rng = _random.Random(500 + seed)
    dp = rng.choice([2, 3, 4])
    cfg.update(dp=dp, layout="shard", ranks=[0], steps=2, grad_scale=1.0, remote_sumsq=0.0, inf_at=None)
    hc_all = H.HostCase(dict(cfg, ranks="all", layout="full"))
    D = H.dopt()
    ranks = []
    for r in range(dp):
        hc = H.HostCase(dict(cfg, ranks=[r]))
        dc = H.DeviceCase(hc)
        wsb = D.dopt_workspace_bytes_bucketed(hc.pm, r)
        ranks.append(dict(hc=hc, dc=dc, wsb=wsb, ws=torch.empty(wsb, dtype=torch.uint8, device="cuda"),
                          local=torch.zeros(1, dtype=torch.float64, device="cuda"),
                          flag=torch.zeros(1, dtype=torch.int32, device="cuda")))
    t_applied = 0
    for t_step in range(1, cfg["steps"] + 1):
        t = t_applied + 1
        full = hc_all.grads(t_step)
        before = H.snapshot(hc_all)
        ores = hc_all.oracle_step(full, t)
        for r, rk in enumerate(ranks):
            reps = [[rk["dc"]._up(_shard(hc_all, bi, x, r)) for x in g] for bi, g in enumerate(full)]
            rk["args"] = rk["dc"].step_args(reps, t)
            rk["args"].c.workspace, rk["args"].c.workspace_bytes = rk["ws"].data_ptr(), rk["wsb"]
            for bi, buf in enumerate(rk["hc"].om.buffers):
                D.dopt_step_reduce_buckets(rk["args"], bi, 0, len(buf.buckets))
            D.dopt_step_local_stats(rk["args"], rk["local"], rk["flag"])
        glob = torch.stack([rk["local"] for rk in ranks]).sum(0)
        gflag = torch.stack([rk["flag"] for rk in ranks]).amax(0)
        found = []
        for rk in ranks:
            rk["args"].set_global_stats(glob, gflag)
            d_found = torch.zeros(1, dtype=torch.int32, device="cuda")
            d_norm = torch.zeros(1, dtype=torch.float32, device="cuda")
            D.dopt_step_finalize(rk["args"], d_found, d_norm)
            for bi, buf in enumerate(rk["hc"].om.buffers):
                D.dopt_step_update_buckets(rk["args"], bi, 0, len(buf.buckets))
            torch.cuda.synchronize()
            found.append((bool(d_found.item()), float(d_norm.item())))
        assert all(f == ores["found_inf"] for f, _ in found), (found, ores["found_inf"])
        if ores["found_inf"]:
            continue
        for _, n in found:
            assert abs(n - ores["norm"]) <= 1e-5 * ores["norm"], (n, ores["norm"])
        for r, rk in enumerate(ranks):
            params, master, exp_avg, exp_avg_sq, _ = rk["dc"].download()
            for bi, buf in enumerate(hc_all.om.buffers):
                S = hc_all.om.shard_numel(bi)
                sl = slice(r * S, (r + 1) * S)
                mask = hc_all.piece_mask(bi)[sl]
                st = hc_all.state[bi]
                for name, got in (("exp_avg", exp_avg[bi]), ("exp_avg_sq", exp_avg_sq[bi]), ("master", master[bi])):
                    if got is None:
                        continue
                    assert H.state_close(got[mask], st[name][sl][mask], before[bi][name][sl][mask]).all(), \
                        (seed, t_step, r, bi, name)
        t_applied += 1
