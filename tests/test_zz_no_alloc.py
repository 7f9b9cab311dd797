"""The allocation-free fused step (dopt_step_noalloc) against the regular one.

dopt_step_noalloc serves callers that cannot allocate device memory -- a
program whose GPU memory belongs to another allocator, a loop that forbids
allocation after start-up, or a plugin interface that passes only inputs and
outputs.  Its scratch is a static device array inside the library instead of
a caller workspace.  These tests call it through the C ABI twice in a row and
check every output against dopt_step's on identical inputs, within the
tolerances the parity tests use, and check that requests larger than the
static scratch are refused.  This file is collected last on purpose.
"""

import numpy as np
import pytest

from synth import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gpu_harness as H  # noqa: E402


def _compare(a, b, before):
    """a, b: DeviceCase after the same step; before: b's arrays before it."""
    pa, ma, ea, va, mna = a.download()
    pb, mb, eb, vb, mnb = b.download()
    for bi in range(len(pa)):
        for g, w, bf in ((ma[bi], mb[bi], before[1][bi]), (ea[bi], eb[bi], before[2][bi]),
                         (va[bi], vb[bi], before[3][bi]), (mna[bi], mnb[bi], before[4][bi])):
            if g is not None:
                assert H.state_close(g, w, bf).all()
        if pa[bi].dtype == np.uint16:
            assert H.ulp16(pa[bi], pb[bi]).max() <= 1
        else:
            assert H.state_close(pa[bi], pb[bi], before[0][bi]).all()


@pytest.mark.parametrize("name", ["llama_7b_dp8_rank0", "gpt2_small_dp8"])
def test_noalloc_matches_dopt_step_two_calls(name):
    D = H.dopt()
    hc = H.HostCase(W.mini(name))
    with_ws = H.DeviceCase(hc)
    no_ws = H.DeviceCase(hc)
    t_applied = 0
    for step in (1, 2):
        grads = hc.grads(step)
        t = t_applied + 1
        before = with_ws.download()
        reps_a = [[no_ws._up(r) for r in g] for g in grads]
        reps_b = [[with_ws._up(r) for r in g] for g in grads]
        args_a = no_ws.step_args(reps_a, t)
        args_a.c.workspace = None  # ignored by the allocation-free entry point
        args_a.c.workspace_bytes = 0
        found_a, norm_a = D.dopt_step_noalloc(args_a)
        found_b, norm_b = D.dopt_step(with_ws.step_args(reps_b, t))
        assert found_a == found_b
        if not found_b:
            assert abs(norm_a - norm_b) <= 1e-5 * norm_b
            t_applied += 1
        _compare(no_ws, with_ws, before)


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
