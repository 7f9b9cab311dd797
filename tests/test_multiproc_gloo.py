"""Multi-process tests on CPU (gloo, world size 2).

1. The benchmark's whole-job aggregation: every rank's elements over the
   slowest rank's time, taken with a MAX all-reduce.
2. The multi-rank composition of the sharded step: each process owns one DP
   rank's shard (its param pieces from the library's shard map), computes its
   main grads and local sum of squares, all-reduces the two step scalars
   (sum of squares and the non-finite flag) and finishes the step with them
   as the remote terms.  The union of the ranks' updated shards must equal
   the single-process step over all ranks (the norm's summation order is the
   only difference).  Also a rank that sees an inf makes every rank skip.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _init(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _aggregate_worker(rank, world, port, out):
    import bench
    _init(rank, world, port)
    elapsed = [100.0, 250.0][rank]
    value, slowest = bench.aggregate(elapsed, 1_000_000, 10, world)
    # the re-measure decision: one rank's bad clock record decides for all
    again = bench.any_rank(rank == 1, world)
    never = bench.any_rank(False, world)
    out[rank] = (value, slowest, again, never)
    dist.destroy_process_group()


def test_bench_aggregate_max_over_ranks():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_aggregate_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for r in (0, 1):
        value, slowest, again, never = res[r]
        assert again is True and never is False
        assert slowest == 250.0
        assert value == pytest.approx(1_000_000 * 10 * 2 / 0.25)


def _case(inject_inf_rank=None):
    from synth import workloads as W
    import synth
    import oracle
    cfg = W._cfg(name="gloo", params=W.llama(1, 64, 172, 101), dp=2, bucket_size=3000, seed=31)
    om = oracle.ShardMap(cfg["params"], 2, cfg["bucket_size"], True)
    grads, params, masters = [], [], []
    pkey = synth.key(cfg["seed"], synth.STREAM_PARAM, 0, 0)
    for bi, buf in enumerate(om.buffers):
        kind = {0: synth.OUT_F32, 1: synth.OUT_BF16}[buf.grad_dtype]
        reps = [synth.normal(buf.numel, synth.key(cfg["seed"], synth.STREAM_GRAD, 1, k), 0, 1e-2, kind)
                for k in range(2)]
        grads.append(reps)
        pk = {0: synth.OUT_F32, 1: synth.OUT_BF16}[buf.param_dtype]
        params.append(synth.normal(buf.numel, pkey, 0, 0.02, pk))
        masters.append(synth.normal(buf.numel, pkey, 0, 0.02, synth.OUT_F32_OF_BF16)
                       if buf.param_dtype != 0 else None)
    if inject_inf_rank is not None:
        # an inf in an element that only rank `inject_inf_rank` owns
        (_, _, v) = om.rank_pieces(0, inject_inf_rank)[0]
        grads[0][1][v["gbuf_world"].start] = np.float32(np.inf)
    return cfg, om, grads, params, masters


def _state_for(om, ranks, masters):
    state = []
    for bi, buf in enumerate(om.buffers):
        S = om.shard_numel(bi)
        st = {"exp_avg": np.zeros(len(ranks) * S, np.float32),
              "exp_avg_sq": np.zeros(len(ranks) * S, np.float32)}
        if masters[bi] is not None:
            ms = np.zeros(len(ranks) * S, np.float32)
            for slot, r in enumerate(ranks):
                for b in range(len(buf.buckets)):
                    rg = om.bucket_world_range(bi, b, r)
                    base = slot * S + om.bucket_shard_base(bi, b)
                    ms[base:base + rg.size] = masters[bi][rg.start:rg.end]
            st["master"] = ms
        state.append(st)
    return state


def _compose_worker(rank, world, port, inject, out):
    import oracle
    import mixed_precision_adam_gb300 as D
    _init(rank, world, port)
    cfg, om, grads, params, masters = _case(inject)
    # this rank's pieces, from the library's shard map (host side of the ABI)
    pm = D.dopt_build_shard_map(cfg["params"], 2, cfg["bucket_size"], True)
    for bi in range(len(om.buffers)):
        got = [(p["param"], p["gbuf_world"]) for p in D.dopt_rank_shards(pm, bi, rank)]
        want = [(pid, v["gbuf_world"].as_tuple()) for pid, _, v in om.rank_pieces(bi, rank)]
        assert got == want
    # phase 1: local main grads and the two local step scalars
    probe = _state_for(om, [rank], masters)
    local = oracle.step(om, [rank], grads, probe, [p.copy() for p in params], cfg["hp"], 1,
                        max_norm=cfg["max_norm"])
    scal = torch.tensor([local["sumsq"], 1.0 if local["found_inf"] else 0.0], dtype=torch.float64)
    tot = scal.clone()
    dist.all_reduce(tot[:1], op=dist.ReduceOp.SUM)
    dist.all_reduce(tot[1:], op=dist.ReduceOp.MAX)
    remote_sumsq = float(tot[0] - scal[0])
    remote_found = bool(tot[1] > 0)
    # phase 2: the step with the other ranks' contribution as remote terms
    state = _state_for(om, [rank], masters)
    res = oracle.step(om, [rank], grads, state, params, cfg["hp"], 1, max_norm=cfg["max_norm"],
                      remote_sumsq=max(remote_sumsq, 0.0), remote_found_inf=remote_found)
    out[rank] = (res["found_inf"], res["norm"], [{k: v.copy() for k, v in s.items()} for s in state],
                 [p.copy() for p in params])
    dist.destroy_process_group()


@pytest.mark.parametrize("inject", [None, 1])
def test_two_rank_composition_matches_single_process(inject):
    import oracle
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_compose_worker, args=(2, port, inject, out), nprocs=2, join=True)
        res = dict(out)
    cfg, om, grads, params, masters = _case(inject)
    state = _state_for(om, [0, 1], masters)
    ref = oracle.step(om, [0, 1], grads, state, params, cfg["hp"], 1, max_norm=cfg["max_norm"])
    for r in (0, 1):
        found, norm, st_r, params_r = res[r]
        assert found == ref["found_inf"]
        if found:
            continue
        assert abs(norm - ref["norm"]) <= 1e-12 * ref["norm"]
        for bi, buf in enumerate(om.buffers):
            S = om.shard_numel(bi)
            for k in st_r[bi]:
                np.testing.assert_array_equal(st_r[bi][k], state[bi][k][r * S:(r + 1) * S])
            for _, _, v in om.rank_pieces(bi, r):
                a, b = v["gbuf_world"].start, v["gbuf_world"].end
                assert params_r[bi][a:b].tobytes() == params[bi][a:b].tobytes()
