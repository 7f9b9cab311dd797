"""The allocation-free fused step (dopt_step_noalloc) against the regular one
and against the oracle.

dopt_step_noalloc serves callers that cannot allocate device memory -- a
program whose GPU memory belongs to another allocator, a loop that forbids
allocation after start-up, or a plugin interface that passes only inputs and
outputs.  Its scratch is a static device array inside the library instead of
a caller workspace.  It runs the same kernels as dopt_step on the same
inputs, so every output must be bit-identical to dopt_step's; each step is
also compared with the oracle at the parity tolerances.  The cases call it
through the C ABI on consecutive steps, through a skipped step right after
a clean one, after a call whose larger map left more filled slots in the
static array than the next map uses, and with a request larger than the
array (refused).  This file is collected last on purpose.
"""

import math

import numpy as np
import pytest

from synth import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gpu_harness as H  # noqa: E402


def _same_bits(a, b):
    for x, y in zip(a, b):
        for u, v in zip(x, y):
            if (u is None) != (v is None):
                return False
            if u is not None and u.tobytes() != v.tobytes():
                return False
    return True


def _same_result(ra, rb):
    (fa, na), (fb, nb) = ra, rb
    if fa != fb:
        return False
    return (math.isnan(na) and math.isnan(nb)) or np.float32(na).tobytes() == np.float32(nb).tobytes()


class _Pair:
    """One workload on the host (oracle) and twice on the device: case a is
    stepped by dopt_step_noalloc, case b by dopt_step."""

    def __init__(self, cfg):
        self.hc = H.HostCase(cfg)
        self.a = H.DeviceCase(self.hc)
        self.b = H.DeviceCase(self.hc)

    def step(self, step, inf_site=None):
        D = H.dopt()
        hc = self.hc
        grads = hc.grads(step)
        if inf_site is not None:  # (buffer, buffer index): +inf in replica 1
            H.plant(hc, grads, inf_site[0], 1, inf_site[1], float("inf"))
        t = hc.t_applied + 1
        before = H.snapshot(hc)
        dev_before = self.a.download()
        ores = hc.oracle_step(grads, t)
        args_a = self.a.step_args([[self.a._up(r) for r in g] for g in grads], t)
        args_a.c.workspace = None  # ignored by the allocation-free entry point
        args_a.c.workspace_bytes = 0
        ra = D.dopt_step_noalloc(args_a)
        rb = D.dopt_step(self.b.step_args([[self.b._up(r) for r in g] for g in grads], t))
        torch.cuda.synchronize()
        assert _same_result(ra, rb), (ra, rb)
        got_a, got_b = self.a.download(), self.b.download()
        assert _same_bits(got_a, got_b), "dopt_step_noalloc and dopt_step differ"
        report = []
        ok = H.compare_step(hc, self.a, ores, ra[0], ra[1], before, report, ws=False)
        ok &= H.compare_step(hc, self.b, ores, rb[0], rb[1], before, report)
        assert ok, "\n".join(report)
        if ra[0]:
            # a skipped step leaves master, m, v and params bit-identical
            for k in (0, 1, 2, 3):
                assert _same_bits([got_a[k]], [dev_before[k]]), k
        else:
            hc.t_applied += 1
        return ra


@pytest.mark.parametrize("name", ["llama_7b_dp8_rank0", "gpt2_small_dp8"])
def test_noalloc_bit_identical_and_oracle_exact_through_a_skip(name):
    cfg = W.mini(name)
    pair = _Pair(cfg)
    site = None
    if cfg.get("inf_at") is None:  # plant one in a param element of the rank's shard
        sites = H.plant_sites(pair.hc)
        site = sites[len(sites) // 2]
    found = [pair.step(s, site if s == 2 else None)[0] for s in (1, 2, 3)]
    assert found == [False, True, False]  # the skipped step comes right after a clean one


def test_noalloc_after_a_larger_map_reads_no_stale_slot():
    """A map of 5,000 params whose alternating weight-decay multipliers keep
    every param its own run needs six launch regions of partial slots; its
    call leaves all of them filled.  The next call's map needs two regions
    (one per buffer): its grad norm and updates must still equal dopt_step's
    bit for bit and the oracle's at the parity tolerances, so nothing it
    read was left over."""
    big = W._cfg(name="many_runs", params=[dict(name=f"p{i}", numel=64 + (i % 3), dtype=W.BF16,
                                                 wd_mult=float(i % 2)) for i in range(5000)],
                 dp=1, bucket_size=None, steps=1, seed=31, grad_sigma=1.0)
    D = H.dopt()
    pb = _Pair(big)
    assert D.dopt_workspace_bytes(pb.hc.pm, pb.hc.rank_arg) >= 256 + 6 * 1024 * 16
    pb.step(1)
    small = _Pair(W.mini("llama_7b_dp8_rank0"))
    assert D.dopt_workspace_bytes(small.hc.pm, small.hc.rank_arg) <= 256 + 2 * 1024 * 16
    small.step(1)
    small.step(2)


def test_noalloc_rejects_oversized_request():
    D = H.dopt()
    # 64,000 params whose weight-decay multipliers alternate never merge into
    # longer runs: 67 launch chunks need more partial slots than the scratch has
    params = [dict(numel=64, dtype=1, wd_mult=float(i % 2)) for i in range(64_000)]
    pm = D.dopt_build_shard_map(params, 1, -1, True)
    assert D.dopt_workspace_bytes(pm, 0) > D.NOALLOC_SCRATCH_BYTES
    info = D.dopt_buffer_info_get(pm, 0)
    dev = torch.device("cuda")
    n = info["numel"]
    grads = [[torch.zeros(n, dtype=torch.float32, device=dev)]]
    state = [torch.zeros(n, dtype=torch.float32, device=dev) for _ in range(4)]
    param = torch.zeros(n, dtype=torch.int16, device=dev)
    args = D.StepArgs(pm, 0, grads, [state[0]], [state[1]], [state[2]], [state[3]], [param],
                      W.HP, 1, None, 0, stream=torch.cuda.current_stream())
    with pytest.raises(D.DoptError) as e:
        D.dopt_step_noalloc(args)
    assert e.value.status == D.E_SIZE
    assert "static scratch" in str(e.value)
