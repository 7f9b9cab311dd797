"""The pre-reduction grad check (check_for_nan_in_grad / check_for_large_grads:
the largest |g| of every replica in every bucket, before the reduction)
against the CPU oracle, bit for bit, on every K1 kernel: the TMA-staged fp32
reduction, the specialised 16-bit and two-instance reductions, the general
kernel (average_in_collective, odd DP, three instances) and the scalar paths
of unaligned runs and ragged run ends; fused and bucket-staged; with large,
infinite and NaN values planted at run starts, middles and ends.  The rest of
each step is compared with the oracle as in the parity tests."""

import numpy as np
import pytest

from synth import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gpu_harness as H  # noqa: E402

# step 1: finite values of distinct sizes (the step applies); step 2: one
# infinity and one NaN among large values (the step is skipped); step 3: no
# planted value (the table holds the grads' own maxima)
PLANTS = [
    [(i, i, (-1.0) ** i * 3.0 * (i + 1)) for i in range(9)],
    [(0, 1, 7.0), (4, 2, np.inf), (8, 3, -np.inf), (5, 0, np.nan), (2, 5, -11.0)],
    [],
]


def _tiny(params, dp, **kw):
    cfg = W._cfg(name="tiny", params=params, dp=dp, steps=3, seed=kw.pop("seed", 17))
    cfg.update(kw)
    return cfg


RAGGED = [dict(numel=n, dtype=d) for n, d in
          [(1, 1), (63, 1), (65, 1), (1000, 0), (127, 1), (4099, 1), (3, 0), (20001, 1), (129, 2)]]


def _check(cfg, staged_group=None, plants=PLANTS):
    ok, report = H.run_check(cfg, plants, staged_group)
    assert ok, "\n".join(report)


@pytest.mark.parametrize("name", ["llama_7b_dp8_rank0", "gpt2_small_dp8", "llama_1p3b_fp16_dp8",
                                  "llama_7b_dp16_2x8_1m", "toy_mlp_dp4"])
def test_workload_mini(name):
    _check(W.mini(name))


def test_bf16_replicas():
    cfg = W.mini("llama_7b_dp8_rank0")
    cfg.update(grad_reduce_in_fp32=False)
    _check(cfg)


@pytest.mark.parametrize("dp", [1, 3, 8])
@pytest.mark.parametrize("grad_fp32", [True, False])
def test_ragged_params(dp, grad_fp32):
    _check(_tiny(RAGGED, dp, bucket_size=5000, grad_reduce_in_fp32=grad_fp32, grad_sigma=1e-2))


def test_general_kernel_average_and_instances():
    params = W.llama(1, 128, 344, 257)
    _check(_tiny(params, 4, bucket_size=20000, average=True))
    _check(_tiny(params, 4, bucket_size=20000, n_inst=3, average=True, layout="shard", ranks=[2]))
    _check(_tiny(params, 4, bucket_size=20000, n_inst=2, grad_reduce_in_fp32=False))


def test_unaligned_runs():
    params = [dict(numel=n, dtype=1) for n in (100, 37, 300, 5, 77)]
    _check(_tiny(params, 32, bucket_size=64))


def test_every_rank_of_shard_layout():
    params = W.llama(1, 96, 256, 131)
    for r in range(4):
        _check(_tiny(params, 4, bucket_size=9000, layout="shard", ranks=[r], steps=3))


def test_empty_rank_leaves_zeros():
    # ranks 1..7 own only padding of the 128-element bucket of a 10-element param
    params = [dict(numel=10, dtype=1), dict(numel=300, dtype=0)]
    _check(_tiny(params, 8, bucket_size=None, layout="shard", ranks=[5]), plants=[[], []])


@pytest.mark.parametrize("name,group", [("llama_7b_dp8_rank0", 1), ("gpt2_small_dp8", 2),
                                        ("llama_7b_dp16_2x8_1m", 3)])
def test_bucket_staged(name, group):
    _check(W.mini(name), staged_group=group)


def test_check_off_leaves_step_unchanged():
    """The same step with and without the check gives identical state."""
    cfg = W.mini("llama_7b_dp8_rank0")
    hc = H.HostCase(cfg)
    plain, checked = H.DeviceCase(hc), H.DeviceCase(hc)
    D = H.dopt()
    amax = torch.zeros((hc.n_rep, D.dopt_total_buckets(hc.pm)), dtype=torch.float32, device="cuda")
    for step in range(1, 3):
        grads = hc.grads(step)
        r1 = plain.step(grads, step)
        args = checked.step_args([[checked._up(r) for r in g] for g in grads], step)
        args.set_grad_check(amax)
        r2 = D.dopt_step(args)
        assert r1 == r2
        for a, b in zip(plain.download(), checked.download()):
            for x, y in zip(a, b):
                if x is not None:
                    assert x.tobytes() == y.tobytes()
        assert float(amax.max()) > 0


def test_misaligned_table_is_refused():
    cfg = W.mini("toy_mlp_dp4")
    hc = H.HostCase(cfg)
    dc = H.DeviceCase(hc)
    D = H.dopt()
    buf = torch.zeros(hc.n_rep * D.dopt_total_buckets(hc.pm) + 1, dtype=torch.float32, device="cuda")
    args = dc.step_args([[dc._up(r) for r in g] for g in hc.grads(1)], 1)
    args.c.grad_amax = buf.data_ptr() + 2
    with pytest.raises(D.DoptError) as e:
        D.dopt_step(args)
    assert e.value.status == D.E_ALIGN
