"""CPU tests of the product library's host side: it loads without a GPU,
exports every symbol of include/dopt.h, builds the same shard map as the
oracle (bit-exact), reproduces the pages' memory and communication
arithmetic, and rejects bad arguments with status codes."""

import json
import os
import random
import re

import numpy as np
import pytest
import torch

import oracle
from synth import workloads as W

dopt = pytest.importorskip("mixed_precision_adam_gb300")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


DEBUG_BLOCK = re.compile(r"#if defined\(DOPT_BOUNDS_CHECK\) && DOPT_BOUNDS_CHECK\n(.*?)#endif", re.S)


def _header_functions(debug_build):
    """Functions include/dopt.h declares for the release build, or (debug_build)
    for the bounds-checked debug build, which adds its test hooks."""
    src = open(os.path.join(ROOT, "include", "dopt.h")).read()
    if not debug_build:
        src = DEBUG_BLOCK.sub("", src)
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dopt_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    debug = os.path.basename(dopt.LIB_PATH) == "libdopt_checked.so"
    names = _header_functions(debug)
    assert len(names) >= 20
    import ctypes
    lib = ctypes.CDLL(dopt.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(dopt.exported_symbols())
    hooks = set(_header_functions(True)) - set(_header_functions(False))
    assert hooks == {"dopt_debug_starve_copy"}
    if not debug:  # the release library carries no test hook
        for n in hooks:
            assert not hasattr(lib, n), n


def _compare_maps(params, dp, bucket_size, grad_fp32, busbw):
    om = oracle.ShardMap(params, dp, None if bucket_size < 0 else bucket_size, grad_fp32, busbw)
    pm = dopt.dopt_build_shard_map(params, dp, bucket_size, grad_fp32, busbw)
    assert dopt.dopt_num_buffers(pm) == len(om.buffers)
    # the grad-check table index: buckets numbered across buffers in order
    assert dopt.dopt_total_buckets(pm) == sum(len(b.buckets) for b in om.buffers)
    for bi, ob in enumerate(om.buffers):
        for k in range(len(ob.buckets)):
            assert dopt.dopt_bucket_number(pm, bi, k) == oracle.bucket_number(om, bi, k)
    for bi, ob in enumerate(om.buffers):
        info = dopt.dopt_buffer_info_get(pm, bi)
        assert (info["param_dtype"], info["grad_dtype"], info["numel"], info["numel_unpadded"],
                info["n_buckets"], info["shard_numel"]) == \
            (ob.param_dtype, ob.grad_dtype, ob.numel, ob.numel_unpadded, len(ob.buckets),
             om.shard_numel(bi))
        for k, bk in enumerate(ob.buckets):
            pb = dopt.dopt_bucket_info_get(pm, bi, k)
            assert (pb["offset"], pb["numel"], pb["numel_unpadded"], pb["shard_base"]) == \
                (bk.offset, bk.numel, bk.numel_unpadded, om.bucket_shard_base(bi, k))
        for pid in ob.params:
            assert dopt.dopt_param_index(pm, pid) == (bi,) + tuple(ob.index[pid])
        for r in range(dp):
            got = dopt.dopt_rank_shards(pm, bi, r)
            want = om.rank_pieces(bi, r)
            assert len(got) == len(want)
            for g, (pid, b, v) in zip(got, want):
                assert (g["param"], g["bucket"], g["rank"]) == (pid, b, r)
                assert g["gbuf_world"] == v["gbuf_world"].as_tuple()
                assert g["gbuf_world_in_bucket"] == v["gbuf_world_in_bucket"].as_tuple()
                assert g["gbuf_local"] == v["gbuf_local"].as_tuple()
                assert g["param_range"] == v["param"].as_tuple()
                assert g["shard_offset"] == v["shard_offset"]


@pytest.mark.parametrize("seed", range(60))
def test_shard_map_matches_oracle_random(seed):
    rng = random.Random(1000 + seed)
    params = [dict(numel=rng.randint(0 if rng.random() < 0.05 else 1, 400),
                   dtype=rng.choice([0, 1, 2]), new_bucket=rng.random() < 0.1,
                   wd_mult=rng.choice([1.0, 0.0])) for _ in range(rng.randint(1, 14))]
    dp = rng.choice([1, 2, 3, 4, 5, 8, 16])
    bucket_size = rng.choice([-1, rng.randint(1, 3000)])
    _compare_maps(params, dp, bucket_size, rng.random() < 0.5, rng.random() < 0.2)


@pytest.mark.parametrize("name", ["toy_mlp_dp4", "gpt2_small_dp8", "llama_1p3b_fp16_dp8",
                                  "llama_7b_dp8_rank0", "llama_7b_dp16_2x8_1m",
                                  "llama_7b_dp16_2x8_100m"])
def test_shard_map_matches_oracle_workloads(name):
    c = W.config(name)
    _compare_maps(c["params"], c["dp"], c["bucket_size"], c["grad_reduce_in_fp32"], False)


def test_default_bucket_size():
    # default bucket size max(40M, 1M * DP): three 30M params; with DP=8
    # (40M) the bucket seals at 60M, leaving a tail bucket; with DP=64 (64M)
    # it seals only at 90M
    params = [dict(numel=30_000_000, dtype=1)] * 3
    m64 = dopt.dopt_build_shard_map(params, 64, 0)
    assert dopt.dopt_buffer_info_get(m64, 0)["n_buckets"] == 1
    m8 = dopt.dopt_build_shard_map(params, 8, 0)
    assert dopt.dopt_buffer_info_get(m8, 0)["n_buckets"] == 2


def test_memory_ledger_matches_pages():
    g = json.load(open(os.path.join(GOLDEN, "memory_ledger.json")))
    c0, c1, c2, c3 = g["cases"]
    # 7B, DP=8: 84 GB of Adam state replicated, 10.5 GB sharded, 73.5 GB (87.5 %) saved
    _, ddp = dopt.dopt_memory_ledger(c0["P"], c0["N"], 0)
    _, z1 = dopt.dopt_memory_ledger(c0["P"], c0["N"], 1)
    assert sum(ddp[2:]) == c0["optimizer_state_bytes"]["ddp"]
    assert sum(z1[2:]) == c0["optimizer_state_bytes"]["zero1"]
    assert sum(ddp[2:]) - sum(z1[2:]) == c0["saved_bytes"]
    assert (sum(ddp[2:]) - sum(z1[2:])) / sum(ddp[2:]) == c0["saved_frac"]
    # 4.375B per card, DP=8: the formula values (the page prints ~26 GB for
    # ZeRO-1, an arithmetic slip of its own: 70 - 45.9 = 24.1)
    for stage, key in enumerate(["ddp", "zero1", "zero2", "zero3"]):
        total, _ = dopt.dopt_memory_ledger(c1["P"], c1["N"], stage)
        assert total == c1["total_bytes"][key]
        assert abs(total / 1e9 - c1["page_printed_gb"][key]) <= (2.0 if key == "zero1" else 0.6)
    # DeepSpeed 7.5B, ZeRO-2 on 8 GPUs: 15 + 1.875 + 11.25 = 28.125 GB
    total, parts = dopt.dopt_memory_ledger(c2["P"], c2["N"], 2)
    assert parts[0] == c2["zero2_parts_bytes"]["param"]
    assert parts[1] == c2["zero2_parts_bytes"]["grad"]
    assert sum(parts[2:]) == c2["zero2_parts_bytes"]["optimizer_state"]
    assert total == c2["zero2_total_bytes"]
    # N=64: 12P -> 12P/64
    _, z64 = dopt.dopt_memory_ledger(c3["P"], c3["N"], 1)
    assert sum(z64[2:]) == c3["optimizer_state_bytes"]["zero1"]
    # the table's general formulas
    for P, N in ((7_000_000_000, 8), (1 << 30, 64), (4096, 1)):
        assert dopt.dopt_memory_ledger(P, N, 0)[0] == 16 * P
        assert dopt.dopt_memory_ledger(P, N, 1)[0] == 4 * P + 12 * P // N
        assert dopt.dopt_memory_ledger(P, N, 2)[0] == 2 * P + 14 * P // N
        assert dopt.dopt_memory_ledger(P, N, 3)[0] == 16 * P // N


def test_comm_conservation():
    # ring reduce-scatter + all-gather = one all-reduce, each about P per rank
    for P, N, b in ((7_000_000_000, 8, 2), (1024, 4, 4), (1000, 3, 2), (5, 8, 2)):
        rs = dopt.dopt_comm_bytes(P, N, b, 0)
        ag = dopt.dopt_comm_bytes(P, N, b, 1)
        ar = dopt.dopt_comm_bytes(P, N, b, 2)
        assert rs == ag and rs + ag == ar
        chunk = -(-P // N)
        assert rs == (N - 1) * chunk * b
    P = 10**9
    assert dopt.dopt_comm_bytes(P, 10**6, 1, 2) / (2 * P) > 0.999


def test_loss_scaler_policy():
    s = dopt.dopt_loss_scaler_init(2.0**16, 2.0, 0.5, growth_interval=3, hysteresis=2)
    assert s.scale == 65536.0
    dopt.dopt_loss_scaler_update(s, True)   # first strike: hysteresis absorbs it
    assert s.scale == 65536.0
    dopt.dopt_loss_scaler_update(s, True)   # second strike: back off
    assert s.scale == 32768.0
    for _ in range(3):
        dopt.dopt_loss_scaler_update(s, False)
    assert s.scale == 65536.0 and s.hysteresis_tracker == 2
    s = dopt.dopt_loss_scaler_init(1.0, 2.0, 0.5, 1000, 1, min_scale=1.0)
    dopt.dopt_loss_scaler_update(s, True)
    assert s.scale == 1.0  # floored at min_scale


def test_bad_arguments_return_status():
    with pytest.raises(dopt.DoptError) as e:
        dopt.dopt_build_shard_map([], 4)
    assert e.value.status == dopt.E_INVALID
    with pytest.raises(dopt.DoptError):
        dopt.dopt_build_shard_map([dict(numel=10, dtype=7)], 4)
    with pytest.raises(dopt.DoptError):
        dopt.dopt_build_shard_map([dict(numel=-1, dtype=1)], 4)
    with pytest.raises(dopt.DoptError):
        dopt.dopt_build_shard_map([dict(numel=10, dtype=1)], 0)
    m = dopt.dopt_build_shard_map([dict(numel=1000, dtype=1)], 4, -1)
    with pytest.raises(dopt.DoptError):
        dopt.dopt_buffer_info_get(m, 5)
    with pytest.raises(dopt.DoptError):
        dopt.dopt_rank_shards(m, 0, 4)
    with pytest.raises(dopt.DoptError):
        dopt.dopt_workspace_bytes(m, 9)
    assert dopt.dopt_workspace_bytes(m, 0) > 0 and dopt.dopt_workspace_bytes(m, dopt.ALL_RANKS) > 0
    with pytest.raises(dopt.DoptError):
        dopt.dopt_memory_ledger(10, 0, 1)
    with pytest.raises(dopt.DoptError):
        dopt.dopt_comm_bytes(10, 2, 2, 7)
    # device entry points validate their arguments before touching the GPU
    ws = dopt.dopt_workspace_bytes(m, 0)
    with pytest.raises(dopt.DoptError) as e:
        dopt.dopt_grad_reduce_shard(m, 0, 0, [16] * 3, 1, dopt.LAYOUT_FULL_BUFFER, False, 16, 16, ws)
    assert e.value.status == dopt.E_INVALID  # 3 replicas for DP=4
    with pytest.raises(dopt.DoptError) as e:
        dopt.dopt_grad_reduce_shard(m, 0, 0, [16, 16, 16, 8], 1, dopt.LAYOUT_FULL_BUFFER, False,
                                    16, 16, ws)
    assert e.value.status == dopt.E_ALIGN
    with pytest.raises(dopt.DoptError) as e:
        dopt.dopt_grad_reduce_shard(m, 0, dopt.ALL_RANKS, [16] * 4, 1, dopt.LAYOUT_SHARD_ONLY,
                                    False, 16, 16, ws)
    assert e.value.status == dopt.E_INVALID
    with pytest.raises(dopt.DoptError) as e:
        dopt.dopt_prepare_grads(m, 0, 0, 1.0, 16, 16, ws - 16)
    assert e.value.status == dopt.E_SIZE
    with pytest.raises(dopt.DoptError) as e:
        dopt.dopt_adam_step(m, 0, 0, 16, 16, 16, 16, 16, W.HP, 0, 16, 16)
    assert e.value.status == dopt.E_INVALID  # step 0
    mf = dopt.dopt_build_shard_map([dict(numel=1000, dtype=0)], 4, -1)
    with pytest.raises(dopt.DoptError) as e:
        dopt.dopt_adam_step(mf, 0, 0, 16, 16, 16, 16, 16, W.HP, 1, 16, 16)
    assert e.value.status == dopt.E_INVALID  # fp32 buffer: master must be NULL

    # model-space state copies: bad buffer, rank, layout or pointer fail
    # before any device work
    pm2 = dopt.dopt_build_shard_map([dict(numel=100, dtype=1), dict(numel=7, dtype=0)], 2, -1, True, False)
    assert [dopt.dopt_model_numel(pm2, b) for b in range(2)] == [100, 7]
    arr = np.zeros(256, np.float32)
    for args in [(2, 0, 0, arr, arr), (0, 2, 0, arr, arr), (0, -2, 0, arr, arr), (0, 0, 5, arr, arr),
                 (0, 0, 0, None, arr), (0, 0, 0, arr, None)]:
        for fn in (dopt.dopt_state_to_model, dopt.dopt_state_from_model):
            with pytest.raises(dopt.DoptError) as e:
                fn(pm2, *args)
            assert e.value.status == dopt.E_INVALID
    # bucket numbering outside the map
    m = dopt.dopt_build_shard_map([dict(numel=100, dtype=1)], 2, -1, True, False)
    for buffer, bucket in [(-1, 0), (1, 0), (0, 1), (0, -1)]:
        with pytest.raises(dopt.DoptError) as e:
            dopt.dopt_bucket_number(m, buffer, bucket)
        assert e.value.status == dopt.E_INVALID


def test_bounds_record_needs_the_checked_build():
    """The default build exports the debug query but refuses it: its kernels
    carry no bounds checks."""
    if os.environ.get("DOPT_LIBRARY"):
        pytest.skip("another build of the library is loaded")
    with pytest.raises(dopt.DoptError) as e:
        dopt.dopt_debug_bounds_record()
    assert e.value.status == dopt.E_INVALID


@pytest.mark.parametrize("growth,backoff,interval,p_inf", [(2.0, 0.5, 1, 0.4), (2.0, 0.5, 3, 0.25),
                                                           (4.0, 0.25, 2, 0.4), (2.0, 0.125, 1, 0.25)])
def test_loss_scaler_with_hysteresis_1_equals_torch_gradscaler_update(growth, backoff, interval, p_inf):
    """With a hysteresis of 1 the dynamic loss scaler reduces to the
    backoff/growth rule of torch's GradScaler (torch._amp_update_scale_, an
    independent library routine): back off on every step with an inf, grow
    after `interval` clean steps in a row.  Same scale and growth counter
    after every step of a seeded random inf pattern (powers of two: exact in
    torch's float32 scale and the library's double; the inf rate keeps the
    scale inside float32's normal range, so the library's min_scale floor,
    which torch lacks, never acts)."""
    rng = random.Random(int(growth * 100 + interval))
    s = dopt.dopt_loss_scaler_init(2.0**16, growth, backoff, interval, 1, min_scale=2.0**-140)
    t_scale = torch.tensor([2.0**16], dtype=torch.float32)
    t_track = torch.tensor([0], dtype=torch.int32)
    for step in range(300):
        found = rng.random() < p_inf
        dopt.dopt_loss_scaler_update(s, found)
        torch._amp_update_scale_(t_scale, t_track, torch.tensor([1.0 if found else 0.0]), growth, backoff,
                                 interval)
        assert s.scale == t_scale.item(), step
        assert s.growth_tracker == t_track.item(), step
        assert 2.0**-126 <= s.scale < 2.0**127


@pytest.mark.parametrize("dp", [2, 8, 64])
def test_rank_buffer_sizes_equal_the_ledger(dp):
    """A bf16 model (2-byte params and grads, as the ledger assumes): what one
    rank holds -- the whole param buffer, its grad buffer (whole in the full
    layout, its shard in the shard-only layout) and the fp32 master, m and v
    of its shard -- is exactly the ledger's ZeRO-1 and ZeRO-2 per-card bytes
    for P = the buffer's size (padding included)."""
    params = [dict(numel=n, dtype=dopt.BF16) for n in (4096 * 4096, 11008 * 4096, 4096, 32000 * 4096)]
    m = dopt.dopt_build_shard_map(params, dp, 0, False, False)  # grads in the param dtype
    assert dopt.dopt_num_buffers(m) == 1
    info = dopt.dopt_buffer_info_get(m, 0)
    P, S = info["numel"], info["shard_numel"]
    assert S * dp == P
    state = 3 * 4 * S                       # master, exp_avg, exp_avg_sq
    zero1 = 2 * P + 2 * P + state           # params + whole grad buffer
    zero2 = 2 * P + 2 * S + state           # params + grad shard
    assert dopt.dopt_memory_ledger(P, dp, 1)[0] == zero1
    assert dopt.dopt_memory_ledger(P, dp, 2)[0] == zero2


def test_bucket_layout_only_for_the_bucket_staged_reduce():
    """DOPT_LAYOUT_BUCKET (replicas that hold one bucket group) is refused,
    before any device work, by every entry point but the bucket-staged
    ones: the fused step, the host-fed step and the separate reduce."""
    m = dopt.dopt_build_shard_map([dict(numel=1000, dtype=1), dict(numel=64, dtype=1, new_bucket=True)],
                                  2, -1, True, False)
    fake = [[16, 32], [48, 64]]  # aligned, never dereferenced
    per_buf = [16, 16]
    ws_fused = dopt.dopt_workspace_bytes(m, 0)
    args = dopt.StepArgs(m, 0, fake, per_buf, per_buf, per_buf, per_buf, per_buf, W.HP, 1, 256, ws_fused,
                         layout=dopt.LAYOUT_BUCKET)
    for call in (lambda: dopt.dopt_step(args), lambda: dopt.dopt_step_async(args, None, None)):
        with pytest.raises(dopt.DoptError) as e:
            call()
        assert e.value.status == dopt.E_INVALID and "bucket" in str(e.value)
    args.c.workspace_bytes = dopt.dopt_workspace_bytes_bucketed(m, 0)
    with pytest.raises(dopt.DoptError) as e:
        dopt.dopt_step_from_host(args, [[np.zeros(4, np.float32)] * 2] * 2)
    assert e.value.status == dopt.E_INVALID and "bucket" in str(e.value)
    with pytest.raises(dopt.DoptError) as e:
        dopt.dopt_grad_reduce_shard(m, 0, 0, [16, 32], 1, dopt.LAYOUT_BUCKET, False, 16, 16,
                                    dopt.dopt_workspace_bytes(m, 0))
    assert e.value.status == dopt.E_INVALID and "bucket" in str(e.value)
    args.c.layout = 7
    with pytest.raises(dopt.DoptError) as e:
        dopt.dopt_step(args)
    assert e.value.status == dopt.E_INVALID
