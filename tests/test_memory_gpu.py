"""The library allocates no device memory: once a first step has run (which
loads the kernels and creates the side stream and event the synchronous
steps copy their results on), further steps leave the device's free memory
unchanged.  A rank's device memory is therefore exactly the buffers its
caller allocates, whose sizes the ledger tests check against the pages'
formulas."""

import pytest

from synth import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gpu_harness as H  # noqa: E402


@pytest.mark.parametrize("name", ["llama_7b_dp8_rank0", "gpt2_small_dp8"])
def test_steps_allocate_no_device_memory(name):
    D = H.dopt()
    cfg = dict(W.mini(name), inf_at=None)
    hc = H.HostCase(cfg)
    dc = H.DeviceCase(hc)
    reps = [[dc._up(r) for r in g] for g in hc.grads(1)]
    args = dc.step_args(reps, 1)
    d_found = torch.zeros(1, dtype=torch.int32, device="cuda")
    d_norm = torch.zeros(1, dtype=torch.float32, device="cuda")
    D.dopt_step(args)  # first step: kernels loaded, side stream and event created
    D.dopt_step_async(args, d_found, d_norm)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for t in range(2, 8):
        args.set_step(t)
        D.dopt_step(args)
        D.dopt_step_async(args, d_found, d_norm)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
