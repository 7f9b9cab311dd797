"""Reshardable optimizer state: dopt_state_to_model / dopt_state_from_model
against a plain gather/scatter over the oracle's shard map, for flat shards
and param buffers, device and host memory, one rank and every rank; and a
run that saves its state at DP=8, restores it at DP=4 (another bucket size,
so another layout) and keeps matching the oracle."""

import numpy as np
import pytest

import oracle
from synth import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gpu_harness as H  # noqa: E402

SENTINEL = -7.0


def _model_start(om, bi):
    out, acc = {}, 0
    for pid in om.buffers[bi].params:
        out[pid] = acc
        acc += om.params[pid]["numel"]
    return out, acc


def _pieces(om, bi, ranks, layout):
    """(state index, model index, length) of the ranks' pieces, from the
    oracle's views: flat shard slot * S + shard_offset, or the buffer index."""
    start, _ = _model_start(om, bi)
    S = om.shard_numel(bi)
    out = []
    for slot, r in enumerate(ranks):
        for pid, _, v in om.rank_pieces(bi, r):
            st = slot * S + v["shard_offset"] if layout == 0 else v["gbuf_world"].start
            out.append((st, start[pid] + v["param"].start, v["gbuf_local"].size))
    return out


def _to_model(om, bi, ranks, layout, state, model):
    for s, m, n in _pieces(om, bi, ranks, layout):
        model[m:m + n] = state[s:s + n]


def _from_model(om, bi, ranks, layout, model, state):
    for s, m, n in _pieces(om, bi, ranks, layout):
        state[s:s + n] = model[m:m + n]


PARAMS = [dict(numel=n, dtype=d) for n, d in
          [(700, 1), (5, 0), (3001, 1), (64, 1), (33, 0), (12000, 1), (129, 2), (1, 1)]]


@pytest.mark.parametrize("dp,bucket", [(8, 2000), (3, None), (4, 700)])
def test_flat_shard_round_trip(dp, bucket):
    D = H.dopt()
    om = oracle.ShardMap(PARAMS, dp, bucket, True)
    pm = D.dopt_build_shard_map(PARAMS, dp, -1 if bucket is None else bucket, True, False)
    for bi in range(len(om.buffers)):
        _, M = _model_start(om, bi)
        assert D.dopt_model_numel(pm, bi) == M
        S = om.shard_numel(bi)
        for ranks, rank_arg in [(list(range(dp)), D.ALL_RANKS), ([dp - 1], dp - 1)]:
            state = np.arange(len(ranks) * S, dtype=np.float32) * np.float32(0.5) + 1
            want = np.full(M, SENTINEL, np.float32)
            _to_model(om, bi, ranks, 0, state, want)
            dev_model = torch.full((M,), SENTINEL, dtype=torch.float32, device="cuda")
            D.dopt_state_to_model(pm, bi, rank_arg, D.STATE_FLAT_SHARD, torch.from_numpy(state).cuda(), dev_model)
            host_model = np.full(M, SENTINEL, np.float32)  # host destination, device source
            D.dopt_state_to_model(pm, bi, rank_arg, D.STATE_FLAT_SHARD, torch.from_numpy(state).cuda(), host_model)
            torch.cuda.synchronize()
            assert np.array_equal(dev_model.cpu().numpy(), want)
            assert np.array_equal(host_model, want)
            # and back, from host model space to device shards with sentinels elsewhere
            back = torch.full((len(ranks) * S,), SENTINEL, dtype=torch.float32, device="cuda")
            D.dopt_state_from_model(pm, bi, rank_arg, D.STATE_FLAT_SHARD, want, back)
            torch.cuda.synchronize()
            expect = np.full(len(ranks) * S, SENTINEL, np.float32)
            _from_model(om, bi, ranks, 0, want, expect)
            assert np.array_equal(back.cpu().numpy(), expect)


def test_param_buffer_16_bit_round_trip():
    D = H.dopt()
    om = oracle.ShardMap(PARAMS, 4, 1500, True)
    pm = D.dopt_build_shard_map(PARAMS, 4, 1500, True, False)
    for bi, buf in enumerate(om.buffers):
        _, M = _model_start(om, bi)
        dt = np.float32 if buf.param_dtype == 0 else np.int16
        pbuf = (np.arange(buf.numel) % 30000).astype(dt)
        want = np.full(M, -3, dt)
        _to_model(om, bi, list(range(4)), 1, pbuf, want)
        got = torch.full((M,), -3, dtype=torch.float32 if dt == np.float32 else torch.int16, device="cuda")
        D.dopt_state_to_model(pm, bi, D.ALL_RANKS, D.STATE_PARAM_BUFFER, torch.from_numpy(pbuf).cuda(), got)
        torch.cuda.synchronize()
        assert np.array_equal(got.cpu().numpy(), want)
        assert not (want == -3).any()  # every param element is some rank's


def test_resume_at_another_dp_matches_oracle():
    """Two steps at DP=8 (all ranks), state saved to model space on the
    device, restored at DP=4 with another bucket size, one more step: the
    oracle, given the same state by the plain scatter, agrees."""
    D = H.dopt()
    params = W.llama(1, 128, 344, 257)
    cfg8 = W._cfg(name="resume8", params=params, dp=8, bucket_size=20000, steps=2, seed=31, warm_state=True)
    hc8 = H.HostCase(cfg8)
    dc8 = H.DeviceCase(hc8)
    report = []
    for step in (1, 2):
        grads = hc8.grads(step)
        before = H.snapshot(hc8)
        ores = hc8.oracle_step(grads, step)
        found, norm = dc8.step(grads, step)
        assert H.compare_step(hc8, dc8, ores, found, norm, before, report), "\n".join(report)
        hc8.t_applied += 1
    ranks8 = list(range(8))
    saved = []  # per buffer: device model-space tensors of master, m, v and the param buffer
    for bi, buf in enumerate(hc8.om.buffers):
        _, M = _model_start(hc8.om, bi)
        rec = {}
        for name, t in [("exp_avg", dc8.exp_avg[bi]), ("exp_avg_sq", dc8.exp_avg_sq[bi]),
                        ("master", dc8.master[bi])]:
            if t is None:
                continue
            rec[name] = torch.empty(M, dtype=torch.float32, device="cuda")
            D.dopt_state_to_model(hc8.pm, bi, D.ALL_RANKS, D.STATE_FLAT_SHARD, t, rec[name])
            want = np.zeros(M, np.float32)
            _to_model(hc8.om, bi, ranks8, 0, hc8.state[bi][name], want)
            assert np.array_equal(rec[name].cpu().numpy(), want), name
        rec["param"] = torch.empty(M, dtype=dc8.params[bi].dtype, device="cuda")
        D.dopt_state_to_model(hc8.pm, bi, D.ALL_RANKS, D.STATE_PARAM_BUFFER, dc8.params[bi], rec["param"])
        saved.append(rec)

    cfg4 = dict(cfg8, name="resume4", dp=4, bucket_size=7000)
    hc4 = H.HostCase(cfg4)
    assert [b.param_dtype for b in hc4.om.buffers] == [b.param_dtype for b in hc8.om.buffers]
    ranks4 = list(range(4))
    for bi in range(len(hc4.om.buffers)):  # the oracle's copy of the restored state
        for name in ("exp_avg", "exp_avg_sq", "master"):
            if name in hc4.state[bi]:
                model = np.zeros(len(saved[bi]["param"]), np.float32)
                _to_model(hc8.om, bi, ranks8, 0, hc8.state[bi][name], model)
                _from_model(hc4.om, bi, ranks4, 0, model, hc4.state[bi][name])
        pmodel = np.zeros(len(saved[bi]["param"]), hc8.params[bi].dtype)
        _to_model(hc8.om, bi, ranks8, 1, hc8.params[bi], pmodel)
        _from_model(hc4.om, bi, ranks4, 1, pmodel, hc4.params[bi])
    dc4 = H.DeviceCase(hc4)  # uploads the restored state ...
    for bi in range(len(hc4.om.buffers)):  # ... which the device restore must reproduce
        for name, t in [("exp_avg", dc4.exp_avg[bi]), ("exp_avg_sq", dc4.exp_avg_sq[bi]),
                        ("master", dc4.master[bi])]:
            if t is None:
                continue
            expect = t.clone()
            t.fill_(SENTINEL)
            D.dopt_state_from_model(hc4.pm, bi, D.ALL_RANKS, D.STATE_FLAT_SHARD, saved[bi][name], t)
            mask = torch.from_numpy(hc4.piece_mask(bi)).cuda()
            assert torch.equal(t[mask], expect[mask]), name
            t.copy_(torch.where(mask, t, expect))
        expect = dc4.params[bi].clone()
        D.dopt_state_from_model(hc4.pm, bi, D.ALL_RANKS, D.STATE_PARAM_BUFFER, saved[bi]["param"],
                                dc4.params[bi])
        assert torch.equal(dc4.params[bi], expect)
    hc4.t_applied = 2
    grads = hc4.grads(3)
    before = H.snapshot(hc4)
    ores = hc4.oracle_step(grads, 3)
    found, norm = dc4.step(grads, 3)
    assert H.compare_step(hc4, dc4, ores, found, norm, before, report), "\n".join(report)
