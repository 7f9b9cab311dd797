"""The bucket-staged step (reduce per bucket as grads become ready, one
finalize, AdamW and write-back per bucket in the order the next forward
needs them) against the fused step: the same arithmetic, so the results must
be bit-identical, whatever the grouping of buckets and the streams used."""

import pytest

from synth import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gpu_harness as H  # noqa: E402


@pytest.mark.parametrize("name,group", [("llama_7b_dp8_rank0", 1), ("gpt2_small_dp8", 2),
                                        ("llama_7b_dp16_2x8_1m", 3), ("llama_1p3b_fp16_dp8", 1)])
def test_bucket_staged_equals_fused(name, group):
    cfg = W.mini(name)
    hc = H.HostCase(cfg)
    fused = H.DeviceCase(hc)
    staged = H.DeviceCase(hc)
    streams = [torch.cuda.Stream() for _ in range(3)]
    t_applied = 0
    for step in range(1, 4):
        grads = hc.grads(step)
        t = t_applied + 1
        f1, n1 = fused.step(grads, t)
        reps = [[staged._up(r) for r in g] for g in grads]
        f2, n2 = H.staged_step(staged, reps, t, group, streams)
        assert f1 == f2
        if not f1:
            assert n1 == n2
            t_applied += 1
        for a, b in zip(fused.download(), staged.download()):
            for x, y in zip(a, b):
                if x is not None:
                    assert x.tobytes() == y.tobytes()


def test_bucket_range_validation():
    D = H.dopt()
    hc = H.HostCase(W.mini("llama_7b_dp8_rank0"))
    dc = H.DeviceCase(hc)
    args = dc.step_args([[dc._up(r) for r in g] for g in hc.grads(1)], 1)
    ws = D.dopt_workspace_bytes_bucketed(hc.pm, hc.rank_arg)
    buf = torch.empty(ws, dtype=torch.uint8, device="cuda")
    args.c.workspace = buf.data_ptr()
    args.c.workspace_bytes = ws
    nbk = D.dopt_buffer_info_get(hc.pm, 0)["n_buckets"]
    for first, count in ((-1, 1), (0, 0), (nbk - 1, 2), (nbk, 1)):
        with pytest.raises(D.DoptError) as e:
            D.dopt_step_reduce_buckets(args, 0, first, count)
        assert e.value.status == D.E_INVALID
    args.c.workspace_bytes = ws - 16
    with pytest.raises(D.DoptError) as e:
        D.dopt_step_finalize(args)
    assert e.value.status == D.E_SIZE
