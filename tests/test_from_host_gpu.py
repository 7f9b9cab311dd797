"""The host-fed step (dopt_step_from_host: replica grads in pinned host
memory, copied bucket by bucket on a copy stream while the reduce pass
runs): element by element against the CPU oracle and bit for bit against the
fused step on device-resident replicas, across layouts, rank selections,
grad dtypes, hierarchical instances, a skipped step, the grad check and a
caller-given copy stream."""

import numpy as np
import pytest

from synth import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gpu_harness as H  # noqa: E402


def _pinned(a):
    t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a.copy())
    return t.pin_memory()


def _host_step(dc, grads, t, copy_stream=None, grad_amax=None):
    """One dopt_step_from_host step on DeviceCase dc: device replica buffers
    of the right size (contents overwritten by the library), the bucket-staged
    workspace, host replicas pinned."""
    D = H.dopt()
    hc = dc.hc
    dev_reps = [[torch.empty_like(dc._up(r)) for r in g] for g in grads]
    host = [[_pinned(r) for r in g] for g in grads]
    args = dc.step_args(dev_reps, t)
    ws_bytes = D.dopt_workspace_bytes_bucketed(hc.pm, hc.rank_arg)
    dc.bws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    args.c.workspace = dc.bws.data_ptr()
    args.c.workspace_bytes = ws_bytes
    if grad_amax is not None:
        args.set_grad_check(grad_amax)
    found, norm = D.dopt_step_from_host(args, host, copy_stream)
    return found, norm, dev_reps


def _run(cfg, steps=3, copy_stream=None):
    hc = H.HostCase(cfg)
    dc = H.DeviceCase(hc)
    ref = H.DeviceCase(hc)
    D = H.dopt()
    total = D.dopt_total_buckets(hc.pm)
    report = []
    for step in range(1, steps + 1):
        grads = hc.grads(step)
        t = hc.t_applied + 1
        before = H.snapshot(hc)
        ores = H.oracle.step(hc.om, hc.ranks, grads, hc.state, hc.params, cfg["hp"], t,
                             inv_scale=float(np.float32(1.0 / cfg["loss_scale"])),
                             max_norm=cfg["max_norm"], layout=cfg["layout"], n_inst=cfg["n_inst"],
                             average=cfg["average"], check_grads=True)
        amax = torch.full((hc.n_rep, total), 7.0, dtype=torch.float32, device="cuda")
        found, norm, _ = _host_step(dc, grads, t, copy_stream, amax)
        assert H.amax_equal(amax.cpu().numpy(), ores["grad_amax"])
        fused_ws = dc.ws
        dc.ws = dc.bws
        ok = H.compare_step(hc, dc, ores, found, norm, before, report)
        dc.ws = fused_ws
        assert ok, "\n".join(report)
        f2, n2 = ref.step(grads, t)
        assert f2 == found and (n2 == norm or (np.isnan(n2) and np.isnan(norm)))
        for a, b in zip(dc.download()[:4], ref.download()[:4]):
            for x, y in zip(a, b):
                if x is not None:
                    assert x.tobytes() == y.tobytes()
        if not ores["found_inf"]:
            hc.t_applied += 1


@pytest.mark.parametrize("name", ["llama_7b_dp8_rank0", "gpt2_small_dp8", "llama_1p3b_fp16_dp8",
                                  "llama_7b_dp16_2x8_1m"])
def test_workload_mini(name):
    _run(W.mini(name))


def test_full_layout_single_rank_and_given_copy_stream():
    cfg = W._cfg(name="tiny", params=W.llama(1, 96, 256, 131), dp=4, bucket_size=9000,
                 ranks=[2], steps=2, seed=5)
    _run(cfg, steps=2, copy_stream=torch.cuda.Stream())


def test_bf16_replicas_all_ranks():
    cfg = W._cfg(name="tiny", params=W.llama(1, 128, 344, 257), dp=4, bucket_size=20000,
                 grad_reduce_in_fp32=False, steps=2, seed=6)
    _run(cfg, steps=2)


def test_argument_errors():
    D = H.dopt()
    cfg = W.mini("toy_mlp_dp4")
    hc = H.HostCase(cfg)
    dc = H.DeviceCase(hc)
    grads = hc.grads(1)
    args = dc.step_args([[dc._up(r) for r in g] for g in grads], 1)
    host = [[_pinned(r) for r in g] for g in grads]
    with pytest.raises(D.DoptError) as e:  # the fused workspace is too small for the staged layout
        D.dopt_step_from_host(args, host)
    assert e.value.status == D.E_SIZE
    ws_bytes = D.dopt_workspace_bytes_bucketed(hc.pm, hc.rank_arg)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    args.c.workspace, args.c.workspace_bytes = ws.data_ptr(), ws_bytes
    side = torch.cuda.Stream()  # a copy stream equal to the step's stream is refused
    args.set_stream(side)
    with pytest.raises(D.DoptError) as e:
        D.dopt_step_from_host(args, host, copy_stream=side)
    assert e.value.status == D.E_INVALID
    args.set_stream(torch.cuda.current_stream())
    bad = [list(h) for h in host]
    bad[0][1] = None
    with pytest.raises(D.DoptError) as e:
        D.dopt_step_from_host(args, bad)
    assert e.value.status == D.E_INVALID
