"""Randomized parity: seeded random parameter lists, DP sizes, bucket sizes,
dtype pairs, replica layouts, rank selections, instances, averaging,
scale_gradients, loss scales, remote norm terms and the grad check, each
stepped through the C ABI (fused, separate or bucket-staged) and compared
with the CPU oracle element by element (with the canary guards of the
harness around every device buffer)."""

import random

import numpy as np
import pytest

from synth import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gpu_harness as H  # noqa: E402


def _random_cfg(seed):
    rng = random.Random(7000 + seed)
    params = []
    for _ in range(rng.randint(1, 24)):
        numel = rng.choice([rng.randint(1, 70), rng.randint(70, 3000), rng.randint(3000, 40000)])
        params.append(dict(numel=numel, dtype=rng.choice([0, 1, 1, 2]),
                           new_bucket=rng.random() < 0.1, wd_mult=rng.choice([1.0, 1.0, 0.0, 0.5])))
    dp = rng.choice([1, 2, 3, 4, 8])
    n_inst = rng.choice([1, 1, 1, 2, 3])
    layout = rng.choice(["full", "shard"])
    ranks = [rng.randrange(dp)] if (layout == "shard" or rng.random() < 0.5) else "all"
    grad_fp32 = rng.random() < 0.6
    f16 = any(p["dtype"] == 2 for p in params) and not grad_fp32
    loss_scale = float(2 ** rng.randint(8, 16)) if f16 else 1.0
    cfg = W._cfg(name=f"random{seed}", params=params, dp=dp, n_inst=n_inst, layout=layout, ranks=ranks,
                 grad_reduce_in_fp32=grad_fp32, bucket_size=rng.choice([None, rng.randint(200, 60000)]),
                 pad_for_high_busbw=rng.random() < 0.2, average=rng.random() < 0.3,
                 loss_scale=loss_scale, grad_sigma=1e-2 * loss_scale,
                 max_norm=rng.choice([1.0, 0.05, 0.0]), steps=2, seed=seed,
                 grad_scale=rng.choice([1.0, 1.0, 0.25, 1.0 / 3.0]), warm_state=rng.random() < 0.5)
    return cfg


@pytest.mark.parametrize("seed", range(24))
def test_random_step_matches_oracle(seed):
    cfg = _random_cfg(seed)
    ok, report = H.run_parity(cfg)
    assert ok, f"{cfg['name']}: dp={cfg['dp']} n_inst={cfg['n_inst']} layout={cfg['layout']} " \
               f"ranks={cfg['ranks']}\n" + "\n".join(report)


@pytest.mark.parametrize("seed", range(24, 32))
def test_random_grad_check_matches_oracle(seed):
    cfg = _random_cfg(seed)
    cfg["grad_scale"] = 1.0
    ok, report = H.run_check(cfg, [[(i, i, 5.0 * (i + 1)) for i in range(4)], [(1, 0, np.inf)]])
    assert ok, "\n".join(report)


@pytest.mark.parametrize("seed", range(32, 48))
def test_random_paths_and_odd_dp_match_oracle(seed):
    """Seeded random maps at DP sizes the workloads do not use (5, 6, 7, 12,
    16, 32: uneven equal splits and the general reduce kernel), with remote
    norm terms, stepped through one of the three paths at random -- the
    fused step, the separate entry points, or the bucket-staged step with
    random bucket groups on two side streams."""
    cfg = _random_cfg(seed)
    rng = random.Random(9000 + seed)
    cfg["dp"] = rng.choice([5, 6, 7, 12, 16, 32])
    cfg["n_inst"] = rng.choice([1, 1, 2])
    if cfg["ranks"] != "all":
        cfg["ranks"] = [rng.randrange(cfg["dp"])]
    cfg["remote_sumsq"] = rng.choice([0.0, 0.0, 1e-3, 5.0])
    path = rng.choice(["fused", "separate", "staged"])
    if path == "separate":
        cfg["grad_scale"] = 1.0  # scale_gradients is a step option of the fused and staged paths
    group = rng.choice([1, 2, 5])
    hc = H.HostCase(cfg)
    dc = H.DeviceCase(hc)
    streams = [torch.cuda.Stream() for _ in range(2)]
    report, ok = [], True
    for t_step in range(1, cfg["steps"] + 1):
        grads = hc.grads(t_step)
        t = hc.t_applied + 1
        before = H.snapshot(hc)
        ores = hc.oracle_step(grads, t)
        if path == "fused":
            found, norm = dc.step(grads, t)
        elif path == "separate":
            found, norm = dc.step_separate(grads, t)
        else:
            found, norm = H.staged_step(dc, [[dc._up(r) for r in g] for g in grads], t, group, streams)
        ok &= H.compare_step(hc, dc, ores, found, norm, before, report, compact=path != "separate",
                             ws=dc.bws if path == "staged" else None)
        if not ores["found_inf"]:
            hc.t_applied += 1
    assert ok, f"{cfg['name']}: path={path} dp={cfg['dp']} n_inst={cfg['n_inst']} layout={cfg['layout']} " \
               f"ranks={cfg['ranks']}\n" + "\n".join(report)
