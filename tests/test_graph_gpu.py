"""The fused step with its step counter and learning rate in device memory,
captured once in a CUDA graph and replayed: fresh grads are copied into the
same replica buffers before every replay, the learning rate follows a
schedule through the device value, and a step with an inf must not advance
the device counter.  Every replay must give exactly the state the
host-driven step gives, and both must match the oracle."""

import numpy as np
import pytest

from synth import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gpu_harness as H  # noqa: E402


def _lr(step):
    return 1e-4 * (1.0 + 0.25 * step)


@pytest.mark.parametrize("name", ["llama_7b_dp8_rank0", "gpt2_small_dp8"])
def test_graph_replay_with_device_step_matches_host_steps(name):
    D = H.dopt()
    cfg = dict(W.mini(name), steps=4, inf_at=None)
    hc = H.HostCase(cfg)
    host = H.DeviceCase(hc)
    graphed = H.DeviceCase(hc)
    warm = H.DeviceCase(hc)  # runs the kernels once outside the capture
    first = hc.grads(1)
    reps = [[graphed._up(r) for r in g] for g in first]
    d_step = torch.zeros(1, dtype=torch.int64, device="cuda")
    d_lr = torch.tensor([_lr(1)], dtype=torch.float64, device="cuda")
    warm_args = warm.step_args([[warm._up(r) for r in g] for g in first], 1)
    warm_d_step = torch.zeros(1, dtype=torch.int64, device="cuda")
    warm_args.set_device_step(warm_d_step, d_lr)
    D.dopt_step_async(warm_args)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        args = graphed.step_args(reps, 1, stream=s)
        args.set_device_step(d_step, d_lr)
        with torch.cuda.graph(graph, stream=s):
            D.dopt_step_async(args)
    torch.cuda.synchronize()

    # the inf of step 2 goes into the first element the first selected rank owns
    _, _, v0 = hc.om.rank_pieces(0, hc.ranks[0])[0]
    inf_at = v0["gbuf_world"].start if cfg["layout"] == "full" else v0["shard_offset"]

    report = []
    for step in range(1, 5):
        grads = hc.grads(step)
        if step == 2:
            g = grads[0][1]
            g[inf_at] = np.inf if g.dtype == np.float32 else 0x7F80
        lr = _lr(step)
        hc.cfg["hp"] = dict(hc.cfg["hp"], lr=lr)
        t = hc.t_applied + 1
        before = H.snapshot(hc)
        ores = hc.oracle_step(grads, t)
        found_h, norm_h = host.step(grads, t)
        assert H.compare_step(hc, host, ores, found_h, norm_h, before, report), "\n".join(report)
        for dst, src in zip(reps, grads):
            for d, h in zip(dst, src):
                d.copy_(torch.from_numpy(h.view(np.int16) if h.dtype == np.uint16 else h))
        d_lr.fill_(lr)
        graph.replay()
        torch.cuda.synchronize()
        stats = D.dopt_read_step_stats(graphed.ws)
        assert bool(stats["found_inf"]) == found_h == (step == 2)
        assert stats["kernel_error"] == 0
        if not found_h:
            hc.t_applied += 1
            assert stats["grad_norm"] == norm_h
        assert int(d_step.item()) == hc.t_applied
        for a, b in zip(host.download(), graphed.download()):
            for x, y in zip(a, b):
                if x is not None:
                    assert x.tobytes() == y.tobytes()


def test_graph_replay_with_grad_check_matches_eager():
    """The grad check inside a captured step (its table is cleared by a
    memset node and merged into with atomic max): every replay gives the
    table an eager step gives, with large and non-finite values planted at
    different places from step to step."""
    D = H.dopt()
    cfg = dict(W.mini("llama_7b_dp8_rank0"), steps=3, inf_at=None)
    hc = H.HostCase(cfg)
    eager = H.DeviceCase(hc)
    graphed = H.DeviceCase(hc)
    warm = H.DeviceCase(hc)
    total = D.dopt_total_buckets(hc.pm)
    sites = H.plant_sites(hc)
    plants = {1: [(0, 0, 9.0), (5, 3, -40.0)], 2: [(2, 1, np.nan), (7, 6, 3.0e4)], 3: [(4, 2, -np.inf)]}

    def grads_of(step):
        g = hc.grads(step)
        for site, k, value in plants[step]:
            bi, w = sites[site % len(sites)]
            H.plant(hc, g, bi, k, w, value)
        return g

    first = grads_of(1)
    reps = [[graphed._up(r) for r in g] for g in first]
    d_step = torch.zeros(1, dtype=torch.int64, device="cuda")
    d_lr = torch.tensor([cfg["hp"]["lr"]], dtype=torch.float64, device="cuda")
    amax_g = torch.zeros((hc.n_rep, total), dtype=torch.float32, device="cuda")
    warm_args = warm.step_args([[warm._up(r) for r in g] for g in first], 1)
    warm_args.set_device_step(torch.zeros(1, dtype=torch.int64, device="cuda"), d_lr)
    warm_args.set_grad_check(torch.zeros_like(amax_g))
    D.dopt_step_async(warm_args)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        args = graphed.step_args(reps, 1, stream=s)
        args.set_device_step(d_step, d_lr)
        args.set_grad_check(amax_g)
        with torch.cuda.graph(graph, stream=s):
            D.dopt_step_async(args)
    torch.cuda.synchronize()

    t_applied = 0
    for step in (1, 2, 3):
        g = first if step == 1 else grads_of(step)
        amax_e = torch.full((hc.n_rep, total), -5.0, dtype=torch.float32, device="cuda")
        eargs = eager.step_args([[eager._up(r) for r in x] for x in g], t_applied + 1)
        eargs.set_grad_check(amax_e)
        found, _ = D.dopt_step(eargs)
        for dst, src in zip(reps, g):
            for d, h in zip(dst, src):
                d.copy_(torch.from_numpy(h.view(np.int16) if h.dtype == np.uint16 else h))
        amax_g.fill_(-5.0)
        graph.replay()
        torch.cuda.synchronize()
        assert H.amax_equal(amax_g.cpu().numpy(), amax_e.cpu().numpy().astype(np.float64)), step
        if not found:
            t_applied += 1
        assert int(d_step.item()) == t_applied
        for a, b in zip(eager.download(), graphed.download()):
            for x, y in zip(a, b):
                if x is not None:
                    assert x.tobytes() == y.tobytes()
