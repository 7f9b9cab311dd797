"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a value the
pages print, a hand-worked example of the pages' rules, a closed form, an
invariant, exact arithmetic, or an independent library routine (numpy,
torch CPU).  None of these tests touches the GPU or the product library.
"""

import json
import math
import os
import random

import numpy as np
import pytest
import torch

import oracle
import synth
from synth import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F32, BF16, F16 = oracle.F32, oracle.BF16, oracle.F16


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# A1 shard map


def test_shard_map_worked_example():
    g = _golden("shard_worked_example.json")
    m = oracle.ShardMap([dict(numel=1024, dtype=BF16)], g["dp"], None)
    (buf,) = m.buffers
    assert len(buf.buckets) == 1 and buf.buckets[0].numel == g["bucket_numel"]
    assert m.shard_numel(0) == g["elements_per_rank"]
    for r, (a, b) in enumerate(g["world_ranges"]):
        assert m.bucket_world_range(0, 0, r).as_tuple() == (a, b)
        (view,) = m.rank_views(0, 0, r).values()
        assert view["param"].as_tuple() == (a, b)
        assert view["gbuf_local"].as_tuple() == (0, 256)


def test_bucketing_hand_worked_cases():
    for case in _golden("bucketing_hand.json")["cases"]:
        nb = case.get("new_bucket", [False] * len(case["numels"]))
        params = [dict(numel=n, dtype=BF16, new_bucket=f) for n, f in zip(case["numels"], nb)]
        m = oracle.ShardMap(params, case["dp"], case["bucket_size"], False, case["busbw"])
        (buf,) = m.buffers
        got = [buf.index[i][:2] for i in range(len(params))]
        assert [list(x) for x in got] == case["param_ranges"], case["why"]
        assert [[b.offset, b.numel, b.numel_unpadded] for b in buf.buckets] == case["buckets"], case["why"]
        # the buffer's sizes: the last bucket's end, and the sum of the
        # buckets' unpadded sizes (the page's final size assertions)
        assert buf.numel == case["buckets"][-1][0] + case["buckets"][-1][1], case["why"]
        assert buf.numel_unpadded == sum(b[2] for b in case["buckets"]), case["why"]


def _random_params(rng, n):
    return [dict(numel=rng.randint(1, 300), dtype=rng.choice([BF16, F16, F32]),
                 new_bucket=rng.random() < 0.1) for _ in range(n)]


@pytest.mark.parametrize("seed", range(40))
def test_shard_map_brute_force_invariants(seed):
    rng = random.Random(seed)
    params = _random_params(rng, rng.randint(1, 12))
    dp = rng.randint(1, 8)
    bucket_size = rng.choice([None, rng.randint(1, 2000)])
    busbw = rng.random() < 0.2
    m = oracle.ShardMap(params, dp, bucket_size, rng.random() < 0.5, busbw)
    divisor = math.lcm(dp, 128, 2**16) if busbw else math.lcm(dp, 128)
    seen_params = set()
    for bi, buf in enumerate(m.buffers):
        assert buf.numel % dp == 0 and buf.numel_unpadded <= buf.numel
        # buckets tile the buffer contiguously, each a multiple of the divisor
        pos = 0
        for bk in buf.buckets:
            assert bk.offset == pos and bk.numel % divisor == 0 and bk.numel_unpadded <= bk.numel
            pos += bk.numel
        assert pos == buf.numel
        # params: 64-aligned starts, inside their bucket's unpadded part, no overlap,
        # laid out in reverse model order
        owner = np.full(buf.numel, -1)
        starts = []
        for pid in buf.params:
            s, e, b = buf.index[pid]
            bk = buf.buckets[b]
            assert s % 64 == 0 and bk.offset <= s and e <= bk.offset + bk.numel_unpadded
            assert (owner[s:e] == -1).all()
            owner[s:e] = pid
            starts.append(s)
            seen_params.add(pid)
        assert starts == sorted(starts, reverse=True)
        # every buffer element has exactly one owning rank: (w - offset) // (numel/dp)
        rank_of = np.full(buf.numel, -1)
        for b, bk in enumerate(buf.buckets):
            for r in range(dp):
                rg = m.bucket_world_range(bi, b, r)
                assert rg.size == bk.numel // dp
                assert (rank_of[rg.start:rg.end] == -1).all()
                rank_of[rg.start:rg.end] = r
            w = np.arange(bk.offset, bk.offset + bk.numel)
            assert (rank_of[w] == (w - bk.offset) // (bk.numel // dp)).all()
        assert (rank_of >= 0).all()
        # per param: the ranks' param views tile [0, numel) exactly once and the
        # four views agree with each other
        cover = {pid: np.zeros(params[pid]["numel"], dtype=int) for pid in buf.params}
        for r in range(dp):
            base = 0
            for b, bk in enumerate(buf.buckets):
                rg = m.bucket_world_range(bi, b, r)
                for pid, v in m.rank_views(bi, b, r).items():
                    s, e, _ = buf.index[pid]
                    gw, gwb, gl, pr = (v["gbuf_world"], v["gbuf_world_in_bucket"],
                                       v["gbuf_local"], v["param"])
                    assert gw.size == gwb.size == gl.size == pr.size > 0
                    assert gw.start - s == pr.start
                    assert gwb.start == gw.start - bk.offset
                    assert gl.start == gw.start - rg.start
                    assert v["shard_offset"] == base + gl.start
                    assert (rank_of[gw.start:gw.end] == r).all()
                    cover[pid][pr.start:pr.end] += 1
                base += bk.numel // dp
        for pid, c in cover.items():
            assert (c == 1).all()
    assert seen_params == set(range(len(params)))


def test_buffers_grouped_by_dtype_pair():
    params = [dict(numel=10, dtype=BF16), dict(numel=10, dtype=F32), dict(numel=10, dtype=BF16)]
    m = oracle.ShardMap(params, 2, None, grad_reduce_in_fp32=False)
    assert [(b.param_dtype, b.grad_dtype, b.params) for b in m.buffers] == \
        [(BF16, BF16, [0, 2]), (F32, F32, [1])]
    m = oracle.ShardMap(params, 2, None, grad_reduce_in_fp32=True)
    assert [(b.param_dtype, b.grad_dtype) for b in m.buffers] == [(BF16, F32), (F32, F32)]


# --------------------------------------------------------------------------
# 16-bit casts: round-to-nearest-even, against numpy / torch


def test_rne_casts_match_libraries():
    rng = np.random.RandomState(0)
    x = np.concatenate([
        (rng.standard_normal(100000) * 0.02).astype(np.float32),
        (rng.standard_normal(20000) * 3e-5).astype(np.float32),
        rng.uniform(-7e4, 7e4, 20000).astype(np.float32),
        np.array([0.0, -0.0, 65504, 65519.996, 65520, 1e-8, 2**-24, 2**-25, 3 * 2**-26,
                  6.1e-5, 2**-14, np.inf, -np.inf, 1e38, -3.4e38], np.float32)])
    bf = oracle.round_bf16(x)
    assert (bf == torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)).all()
    with np.errstate(over="ignore"):
        f16 = x.astype(np.float16).view(np.uint16)
    assert (oracle.round_f16(x) == f16).all()
    # ties to even: 1 + 2^-8 sits halfway between two bf16 values
    assert oracle.round_bf16([1 + 2**-8])[0] == 0x3F80
    assert oracle.round_bf16([1 + 3 * 2**-8])[0] == 0x3F82


def test_casts_keep_nan_a_nan():
    """IEEE: a NaN operand gives a NaN, also when its payload sits only in
    the low bits that the cast drops (which truncation alone would turn into
    an infinity)."""
    nans = np.array([0x7F800001, 0xFF800001, 0x7F80FFFF, 0x7FC00000, 0xFFFFFFFF], np.uint32).view(np.float32)
    for h in oracle.round_bf16(nans):
        assert (h & 0x7F80) == 0x7F80 and (h & 0x007F) != 0, hex(h)
    for h in oracle.round_f16(nans):
        assert (h & 0x7C00) == 0x7C00 and (h & 0x03FF) != 0, hex(h)


# --------------------------------------------------------------------------
# A2 reduce-scatter semantics and A3 prepare


def _exact_replicas(rng, n_rep, n, dtype=np.float32):
    # small integers times 2^-12: every partial sum is exact in fp32, in any order
    return [(rng.randint(-2000, 2000, n) * 2.0**-12).astype(dtype) for _ in range(n_rep)]


@pytest.mark.parametrize("n_rep", [1, 2, 4, 8, 16])
def test_reduce_exact_sum_and_prescale_equals_average(n_rep):
    rng = np.random.RandomState(n_rep)
    reps = _exact_replicas(rng, n_rep, 777)
    exact = np.sum(np.stack(reps).astype(np.float64), axis=0) / n_rep
    out, bad = oracle.reduce_prepare(reps, F32, 0, 777, 1.0)
    assert bad == 0 and (out.astype(np.float64) == exact).all()
    avg, _ = oracle.reduce_prepare(reps, F32, 0, 777, 1.0, average=True)
    assert (avg == out).all()


def test_reduce_hierarchical_matches_flat_on_exact_values():
    rng = np.random.RandomState(7)
    reps = _exact_replicas(rng, 16, 513)
    flat, _ = oracle.reduce_prepare(reps, F32, 0, 513, 1.0)
    for n_inst in (1, 2, 4):
        h, _ = oracle.reduce_prepare(reps, F32, 0, 513, 1.0, n_inst=n_inst)
        assert (h == flat).all()
        ha, _ = oracle.reduce_prepare(reps, F32, 0, 513, 1.0, n_inst=n_inst, average=True)
        assert (ha == flat).all()


def test_reduce_rounds_once_to_grad_dtype():
    rng = np.random.RandomState(3)
    reps32 = [(rng.standard_normal(999) * 1e-3).astype(np.float32) for _ in range(8)]
    for gdt, tdt in ((BF16, torch.bfloat16), (F16, torch.float16)):
        reps = [torch.from_numpy(r).to(tdt) for r in reps32]
        bits = [r.view(torch.int16).numpy().view(np.uint16) for r in reps]
        out, _ = oracle.reduce_prepare(bits, gdt, 0, 999, 1.0)
        # reference: widen exactly, fp32 sum in replica order (each term /8, exact),
        # then one torch cast to the grad dtype
        acc = reps[0].float() * 0.125
        for r in reps[1:]:
            acc = acc + r.float() * 0.125
        want = acc.to(tdt).float().numpy()
        assert (out == want).all()


def test_reduced_grads_are_grad_dtype_values_at_every_level():
    """The reduce-scatter writes into the grad buffer, and the all-reduce
    between instances reduces those buffers: with bf16/fp16 grads the result
    is a value of that dtype at either level, so widening it and casting it
    back to the dtype (torch's cast) changes nothing."""
    rng = np.random.RandomState(5)
    reps32 = [(rng.standard_normal(2000) * 1e-3).astype(np.float32) for _ in range(16)]
    for gdt, tdt in ((BF16, torch.bfloat16), (F16, torch.float16)):
        bits = [torch.from_numpy(r).to(tdt).view(torch.int16).numpy().view(np.uint16) for r in reps32]
        for n_inst in (1, 2, 4):
            for average in (False, True):
                out, _ = oracle.reduce_prepare(bits, gdt, 0, 2000, 1.0, n_inst=n_inst, average=average)
                back = torch.from_numpy(out).to(tdt).float().numpy()
                assert (back == out).all(), (gdt, n_inst, average)


def test_scale_gradients_rounds_once_in_grad_dtype():
    """scale_gradients multiplies the reduced grad in its own dtype: the same
    as torch's in-dtype multiply of the reduced tensor."""
    rng = np.random.RandomState(4)
    reps32 = [(rng.standard_normal(777) * 1e-2).astype(np.float32) for _ in range(4)]
    f = float(np.float32(1.0 / 3.0))
    for gdt, tdt in ((F32, torch.float32), (BF16, torch.bfloat16), (F16, torch.float16)):
        reps = [torch.from_numpy(r).to(tdt) for r in reps32]
        arrs = [r.numpy() if tdt == torch.float32 else r.view(torch.int16).numpy().view(np.uint16)
                for r in reps]
        plain, _ = oracle.reduce_prepare(arrs, gdt, 0, 777, 1.0)
        scaled, _ = oracle.reduce_prepare(arrs, gdt, 0, 777, 0.5, grad_scale=f)
        want = (torch.from_numpy(plain).to(tdt) * f).float() * 0.5
        assert (scaled == want.numpy()).all()
        same, _ = oracle.reduce_prepare(arrs, gdt, 0, 777, 1.0, grad_scale=1.0)
        assert (same == plain).all()


def test_prepare_unscale_and_inf_detection():
    reps = [np.full(64, 65536.0 * 3, np.float32) for _ in range(4)]
    out, bad = oracle.reduce_prepare(reps, F32, 0, 64, 1.0 / 65536)
    assert bad == 0 and (out == 3.0).all()
    for pos in (0, 31, 63):
        for v in (np.inf, -np.inf, np.nan):
            rr = [r.copy() for r in reps]
            rr[2][pos] = v
            _, bad = oracle.reduce_prepare(rr, F32, 0, 64, 1.0)
            assert bad == 1


def test_reduce_sign_of_zero():
    reps = [np.full(8, -0.0, np.float32) for _ in range(4)]
    out, _ = oracle.reduce_prepare(reps, F32, 0, 8, 1.0)
    assert (np.signbit(out)).all()  # -0 + -0 = -0 in IEEE arithmetic


# --------------------------------------------------------------------------
# full step: norm, clip, AdamW, skip


def _setup(params, dp, bucket_size=None, seed=0, layout="full", ranks=None, n_inst=1,
           grad_fp32=True, grad_sigma=1e-3, warm=False):
    m = oracle.ShardMap(params, dp, bucket_size, grad_fp32)
    ranks = list(range(dp)) if ranks is None else ranks
    n_rep = dp * n_inst
    grads, state, pbufs = [], [], []
    for bi, buf in enumerate(m.buffers):
        S = m.shard_numel(bi)
        kind = {F32: synth.OUT_F32, BF16: synth.OUT_BF16, F16: synth.OUT_F16}[buf.grad_dtype]
        n = buf.numel if layout == "full" else S
        grads.append([synth.normal(n, synth.key(seed, synth.STREAM_GRAD, 1, k), 0, grad_sigma, kind)
                      for k in range(n_rep)])
        pkind = {F32: synth.OUT_F32, BF16: synth.OUT_BF16, F16: synth.OUT_F16}[buf.param_dtype]
        pk = synth.key(seed, synth.STREAM_PARAM, 0, 0)
        pbufs.append(synth.normal(buf.numel, pk, 0, 0.02, pkind))
        st = {"exp_avg": np.zeros(len(ranks) * S, np.float32),
              "exp_avg_sq": np.zeros(len(ranks) * S, np.float32)}
        if warm:
            st["exp_avg"] = synth.normal(len(ranks) * S, synth.key(seed, synth.STREAM_EXP_AVG, 0, 0), 0, 1e-4)
            st["exp_avg_sq"] = synth.uniform(len(ranks) * S, synth.key(seed, synth.STREAM_EXP_AVG_SQ, 0, 0), 0, 1e-6)
        if buf.param_dtype != F32:
            full = synth.normal(buf.numel, pk, 0, 0.02,
                                synth.OUT_F32_OF_BF16 if buf.param_dtype == BF16 else synth.OUT_F32_OF_F16)
            master = np.zeros(len(ranks) * S, np.float32)
            for slot, r in enumerate(ranks):
                for b in range(len(buf.buckets)):
                    rg = m.bucket_world_range(bi, b, r)
                    base = slot * S + m.bucket_shard_base(bi, b)
                    master[base:base + rg.size] = full[rg.start:rg.end]
            st["master"] = master
        state.append(st)
    return m, ranks, grads, state, pbufs


def test_norm_closed_form():
    # every main grad equal to c: norm = |c| * sqrt(n); chosen so sqrt is exact
    n = 4**6
    params = [dict(numel=n, dtype=BF16)]
    m = oracle.ShardMap(params, 4, None, True)
    c = 2.0**-7
    grads = [[np.full(n, c, np.float32) for _ in range(4)]]  # avg of 4 equal replicas = c
    st = [{"exp_avg": np.zeros(n, np.float32), "exp_avg_sq": np.zeros(n, np.float32),
           "master": np.zeros(n, np.float32)}]
    res = oracle.step(m, [0, 1, 2, 3], grads, st, [np.zeros(n, np.uint16)], W.HP, 1, max_norm=0.0)
    assert res["norm"] == c * 2**6


def test_norm_matches_library_vector_norm():
    m, ranks, grads, st, pb = _setup(W.toy_mlp(blocks=1, d_in=96, d_hidden=80), 4, 5000)
    res = oracle.step(m, ranks, grads, st, pb, W.HP, 1, max_norm=0.0)
    allm = np.concatenate(res["main"]).astype(np.float64)
    want = torch.linalg.vector_norm(torch.from_numpy(allm)).item()
    assert abs(res["norm"] - want) <= 1e-12 * want


def test_norm_adds_the_remote_sum_of_squares():
    """The norm covers the whole optimizer instance: the remote ranks' sum
    of squares adds under the square root.  Local grads all 2^-7 over 4^6
    elements give 0.25; a remote 0.75 makes the norm exactly 1."""
    n = 4**6
    m = oracle.ShardMap([dict(numel=n, dtype=BF16)], 4, None, True)
    grads = [[np.full(n, 2.0**-7, np.float32) for _ in range(4)]]
    st = [{"exp_avg": np.zeros(n, np.float32), "exp_avg_sq": np.zeros(n, np.float32),
           "master": np.zeros(n, np.float32)}]
    res = oracle.step(m, [0, 1, 2, 3], grads, st, [np.zeros(n, np.uint16)], W.HP, 1,
                      max_norm=0.0, remote_sumsq=0.75)
    assert res["sumsq"] == 1.0 and res["norm"] == 1.0


def _zero_state(m, ranks):
    st, pb = [], []
    for i, b in enumerate(m.buffers):
        n = len(ranks) * m.shard_numel(i)
        st.append({"exp_avg": np.zeros(n, np.float32), "exp_avg_sq": np.zeros(n, np.float32),
                   **({"master": np.zeros(n, np.float32)} if b.param_dtype != F32 else {})})
        pb.append(np.zeros(b.numel, np.uint16 if b.param_dtype != F32 else np.float32))
    return st, pb


def test_count_zeros_counts_main_grads_equal_to_zero():
    """count_zeros counts the stepped main grads equal to zero, +0 or -0.
    Zeros are planted three ways (all replicas +0, all -0, and x / -x that
    cancel exactly after the 1/2 prescale); every other element is nonzero
    and padding is never stepped, so the count is the number of planted
    param elements."""
    params = [dict(numel=n, dtype=d) for n, d in [(70, BF16), (5, F32), (130, BF16), (33, F32)]]
    m = oracle.ShardMap(params, 2, 100, True)
    rng = np.random.RandomState(11)
    grads, want = [], 0
    for buf in m.buffers:
        owned = np.zeros(buf.numel, bool)
        for pid in buf.params:
            s0, e0, _ = buf.index[pid]
            owned[s0:e0] = True
        a = rng.uniform(0.5, 1.5, buf.numel).astype(np.float32)
        r0, r1 = a.copy(), a.copy()
        for w in range(0, buf.numel, 5):
            kind = (w // 5) % 3
            if kind == 0:
                r0[w] = r1[w] = 0.0
            elif kind == 1:
                r0[w] = r1[w] = -0.0
            else:
                r0[w], r1[w] = 0.75, -0.75
            want += int(owned[w])
        grads.append([r0, r1])
    st, pb = _zero_state(m, [0, 1])
    res = oracle.step(m, [0, 1], grads, st, pb, W.HP, 1)
    assert res["num_zeros"] == want and want > 0


def test_zero_grads_with_no_decay_group_leave_params_unchanged():
    """wd_mult scales the decoupled decay per param: with a zero grad, m = v
    = 0 and the update term is 0, so a param with wd_mult 0 keeps its value
    bit for bit while a param with wd_mult 1 decays."""
    params = [dict(numel=300, dtype=BF16, wd_mult=0.0), dict(numel=500, dtype=BF16, wd_mult=1.0)]
    hp = dict(lr=1e-2, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    m = oracle.ShardMap(params, 1, None, True)
    (buf,) = m.buffers
    p0 = synth.normal(buf.numel, synth.key(13, synth.STREAM_PARAM, 0, 0), 0, 0.02, synth.OUT_F32_OF_BF16)
    st = [{"master": p0.copy(), "exp_avg": np.zeros(buf.numel, np.float32),
           "exp_avg_sq": np.zeros(buf.numel, np.float32)}]
    oracle.step(m, [0], [[np.zeros(buf.numel, np.float32)]], st, [np.zeros(buf.numel, np.uint16)], hp, 1)
    s0, e0, _ = buf.index[0]
    s1, e1, _ = buf.index[1]
    assert (st[0]["master"][s0:e0] == p0[s0:e0]).all()
    nz = p0[s1:e1] != 0
    assert (np.abs(st[0]["master"][s1:e1][nz]) < np.abs(p0[s1:e1][nz])).all()


def test_step_dp1_matches_torch_adamw_and_clip():
    """DP=1 is a plain mixed-precision AdamW step: compare with torch's own
    clip_grad_norm_ and AdamW(foreach=False) on CPU fp32 over several steps."""
    params = [dict(numel=3000, dtype=F32), dict(numel=1001, dtype=F32)]
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    m = oracle.ShardMap(params, 1, None, True)
    (buf,) = m.buffers
    p0 = synth.normal(buf.numel, synth.key(5, synth.STREAM_PARAM, 0, 0), 0, 0.02)
    tparams = [torch.nn.Parameter(torch.from_numpy(p0[s:e].copy()))
               for s, e, _ in (buf.index[i] for i in range(2))]
    opt = torch.optim.AdamW(tparams, lr=hp["lr"], betas=(hp["beta1"], hp["beta2"]),
                            eps=hp["eps"], weight_decay=hp["weight_decay"], foreach=False)
    pbuf = p0.copy()
    st = [{"exp_avg": np.zeros(buf.numel, np.float32), "exp_avg_sq": np.zeros(buf.numel, np.float32)}]
    for t in range(1, 6):
        before = pbuf.copy()
        g = synth.normal(buf.numel, synth.key(5, synth.STREAM_GRAD, t, 0), 0, 0.05)
        max_norm = 1.0 if t % 2 else 1e9  # clipped and unclipped branches
        res = oracle.step(m, [0], [[g]], st, [pbuf], hp, t, max_norm=max_norm)
        for i, tp in enumerate(tparams):
            s, e, _ = buf.index[i]
            tp.grad = torch.from_numpy(g[s:e].copy())
        tn = torch.nn.utils.clip_grad_norm_(tparams, max_norm)
        assert abs(res["norm"] - tn.item()) <= 1e-6 * tn.item()
        assert res["clip"] == (t % 2 == 1)
        opt.step()
        for i, tp in enumerate(tparams):
            s, e, _ = buf.index[i]
            # differences carried from earlier steps are absolute, so bound them
            # by ulps of the tensor's scale rather than of each (possibly
            # cancelled, tiny) element
            got, want = pbuf[s:e], tp.detach().numpy()
            tol = 4 * float(np.spacing(np.float32(np.abs(want).max())))
            assert np.abs(got.astype(np.float64) - want).max() <= tol, t
            if t == 1:  # no history yet: element-wise, in ulps of the operands
                assert oracle.master_close(got, want, before[s:e], hp["lr"]).all()
            # torch updates m with lerp (m + w*(g - m)), which rounds differently
            # from beta1*m + (1-beta1)*g; the gap stays at rounding level
            ea = opt.state[tp]["exp_avg"].numpy()
            assert np.abs(st[0]["exp_avg"][s:e] - ea).max() <= 1e-5 * np.abs(ea).max(), t
            va = opt.state[tp]["exp_avg_sq"].numpy()
            assert oracle.float_ulp_diff(st[0]["exp_avg_sq"][s:e], va).max() <= 4, t


def test_step1_closed_form_and_zero_grads():
    """From m = v = 0 the first update is lr * g / (|g| + eps) after the decay
    p * (1 - lr*wd); elements with g = 0 only decay."""
    n = 4096
    params = [dict(numel=n, dtype=BF16)]
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    m = oracle.ShardMap(params, 1, None, True)
    g = synth.normal(n, synth.key(9, synth.STREAM_GRAD, 1, 0), 0, 1e-2)
    g[::7] = 0.0
    p0 = synth.normal(n, synth.key(9, synth.STREAM_PARAM, 0, 0), 0, 0.02, synth.OUT_F32_OF_BF16)
    st = [{"master": p0.copy(), "exp_avg": np.zeros(n, np.float32), "exp_avg_sq": np.zeros(n, np.float32)}]
    pb = np.zeros(n, np.uint16)
    oracle.step(m, [0], [[g]], st, [pb], hp, 1, max_norm=0.0)
    p0d, gd = p0.astype(np.float64), g.astype(np.float64)
    want = p0d * (1 - hp["lr"] * hp["weight_decay"]) - hp["lr"] * gd / (np.abs(gd) + hp["eps"])
    got = st[0]["master"].astype(np.float64)
    assert np.abs(got - want).max() <= 4 * np.spacing(np.float32(0.1))
    z = g == 0
    decay = np.float32(1 - hp["lr"] * hp["weight_decay"])
    assert (st[0]["master"][z] == p0[z] * decay).all()
    assert (st[0]["exp_avg"][z] == 0).all() and (st[0]["exp_avg_sq"][z] == 0).all()
    # the write-back is the RNE cast of the new master (pinned against torch above)
    assert (pb == oracle.round_bf16(st[0]["master"])).all()


@pytest.mark.parametrize("dp", [2, 4, 8])
def test_sharding_invariance(dp):
    """The union of all ranks' shards equals the DP=1 step, up to the norm's
    summation order (coef within 1e-6): the shard map only decides who
    updates an element, not how."""
    params = W.llama(1, 64, 172, 77)
    res = {}
    for d in (1, dp):
        m, ranks, _, st, pb = _setup(params, d, 3000, seed=21)
        grads = []
        for bi, buf in enumerate(m.buffers):
            g = synth.normal(buf.numel, synth.key(21, synth.STREAM_GRAD, 1, 0), 0, 1e-2)
            # replica 0 carries d*g, the others 0: the prescaled sum is exactly g
            grads.append([g * np.float32(d)] + [np.zeros_like(g) for _ in range(d - 1)])
        out = oracle.step(m, ranks, grads, st, pb, W.HP, 1)
        per_param = {}
        for bi, buf in enumerate(m.buffers):
            S = m.shard_numel(bi)
            for slot, r in enumerate(ranks):
                for pid, b, v in m.rank_pieces(bi, r):
                    arr = per_param.setdefault(pid, np.zeros(params[pid]["numel"], np.float32))
                    lo = slot * S + v["shard_offset"]
                    if "master" in st[bi]:
                        piece = st[bi]["master"][lo:lo + v["param"].size]
                    else:
                        piece = pb[bi][v["gbuf_world"].start:v["gbuf_world"].end]
                    arr[v["param"].start:v["param"].end] = piece
        res[d] = (per_param, out["coef"])
    (a, ca), (b, cb) = res[1], res[dp]
    assert ca < 1 and abs(ca - cb) <= 1e-6 * ca
    for pid in a:
        assert oracle.float_ulp_diff(a[pid], b[pid]).max() <= 4


@pytest.mark.parametrize("rank", [1, 3])
def test_shard_only_replicas_equal_the_full_buffers_slice(rank):
    """A shard-only replica holds exactly the rank's slice of every bucket of
    the full grad buffer, concatenated in bucket order: stepping a rank from
    those slices gives the same main grads, state and params as stepping it
    from the full buffers."""
    params = W.gpt2(layers=1, d=64, ffn=256, vocab=97, n_pos=33)
    m, _, grads, st_full, pb_full = _setup(params, 4, 9000, seed=17, ranks=[rank])
    _, _, _, st_shard, pb_shard = _setup(params, 4, 9000, seed=17, ranks=[rank])
    sliced = []
    for bi, buf in enumerate(m.buffers):
        idx = np.concatenate([np.arange(*m.bucket_world_range(bi, b, rank).as_tuple())
                              for b in range(len(buf.buckets))])
        assert idx.size == m.shard_numel(bi)
        sliced.append([g[idx].copy() for g in grads[bi]])
    a = oracle.step(m, [rank], grads, st_full, pb_full, W.HP, 1, layout="full")
    b = oracle.step(m, [rank], sliced, st_shard, pb_shard, W.HP, 1, layout="shard")
    assert a["sumsq"] == b["sumsq"] and a["coef"] == b["coef"]
    for x, y in zip(a["main"], b["main"]):
        assert x.tobytes() == y.tobytes()
    for s0, s1 in zip(st_full, st_shard):
        for k in s0:
            assert s0[k].tobytes() == s1[k].tobytes()
    for p0, p1 in zip(pb_full, pb_shard):
        assert p0.tobytes() == p1.tobytes()
    assert len(m.buffers) == 2 and any(len(buf.buckets) > 1 for buf in m.buffers)


def test_skip_leaves_state_untouched():
    m, ranks, grads, st, pb = _setup(W.gpt2(layers=1, d=64, ffn=256, vocab=97, n_pos=33), 4, 9000,
                                     warm=True)
    before = [{k: v.copy() for k, v in s.items()} for s in st]
    pbefore = [p.copy() for p in pb]
    for bi in range(len(m.buffers)):
        g = grads[bi][1]
        g[len(g) // 2] = np.inf
        res = oracle.step(m, ranks, grads, st, pb, W.HP, 1)
        assert res["found_inf"] and math.isnan(res["norm"])
        for s0, s1 in zip(before, st):
            for k in s0:
                assert s0[k].tobytes() == s1[k].tobytes()
        for p0, p1 in zip(pbefore, pb):
            assert p0.tobytes() == p1.tobytes()
        g[len(g) // 2] = 0.0
    res = oracle.step(m, ranks, grads, st, pb, W.HP, 1, remote_found_inf=True)
    assert res["found_inf"]


def test_inf_anywhere_in_params_skips_but_padding_does_not():
    """Brute force over a tiny two-buffer map with padding: a non-finite grad
    at any param element of any rank's shard sets found_inf; one in a
    padding position is never read (padding is not a parameter)."""
    params = [dict(numel=n, dtype=d) for n, d in [(70, BF16), (5, F32), (130, BF16), (33, F32)]]
    m = oracle.ShardMap(params, 4, 100, True)
    owned = [np.zeros(b.numel, bool) for b in m.buffers]
    for bi, buf in enumerate(m.buffers):
        for pid in buf.params:
            s0, e0, _ = buf.index[pid]
            owned[bi][s0:e0] = True
    assert not all(o.all() for o in owned)  # the map has padding
    for bi, buf in enumerate(m.buffers):
        for w in range(buf.numel):
            grads = [[np.zeros(b.numel, np.float32) for _ in range(4)] for b in m.buffers]
            grads[bi][w % 4][w] = np.inf
            st = [{"exp_avg": np.zeros(4 * m.shard_numel(i), np.float32),
                   "exp_avg_sq": np.zeros(4 * m.shard_numel(i), np.float32),
                   **({"master": np.zeros(4 * m.shard_numel(i), np.float32)}
                      if b.param_dtype != F32 else {})} for i, b in enumerate(m.buffers)]
            pb = [np.zeros(b.numel, np.uint16 if b.param_dtype != F32 else np.float32)
                  for b in m.buffers]
            res = oracle.step(m, [0, 1, 2, 3], grads, st, pb, W.HP, 1)
            assert res["found_inf"] == bool(owned[bi][w]), (bi, w)


# --------------------------------------------------------------------------
# A2 check: largest |g| per replica and bucket before the reduction


def test_grad_amax_run_hand_values():
    """Values fixed by the IEEE / bfloat16 formats: the largest magnitude,
    +inf over any finite value, NaN over everything, 0 for nothing read."""
    f = lambda xs: np.array(xs, np.float32)
    u = lambda xs: np.array(xs, np.uint16)
    amax = oracle.grad_amax_run
    assert amax(f([1.0, -3.5, 2.0, 0.0]), F32, 0, 4) == 3.5
    assert amax(f([-0.0, 0.0]), F32, 0, 2) == 0.0
    assert amax(f([9.0]), F32, 0, 0) == 0.0
    assert amax(f([100.0, 1.0, 2.0, -7.0, 50.0]), F32, 1, 3) == 7.0  # index0 and length
    assert amax(f([1.0, np.inf]), F32, 0, 2) == math.inf
    assert amax(f([-np.inf, 5.0]), F32, 0, 2) == math.inf
    assert math.isnan(amax(f([np.nan, np.inf, 1.0]), F32, 0, 3))
    assert math.isnan(amax(f([1.0, -np.nan]), F32, 0, 2))
    assert amax(f([3.4028235e38, -1.0]), F32, 0, 2) == 3.4028234663852886e38
    # bf16: 0xC0A0 = -5, 0x3F80 = 1, 0x0001 = 2^-133 (smallest subnormal)
    assert amax(u([0x3F80, 0xC0A0]), BF16, 0, 2) == 5.0
    assert amax(u([0x0001, 0x8000]), BF16, 0, 2) == 2.0 ** -133
    assert amax(u([0xFF80, 0x3F80]), BF16, 0, 2) == math.inf
    assert math.isnan(amax(u([0x7FC0, 0x7F80]), BF16, 0, 2))
    # fp16: 0xBC00 = -1, 0x4500 = 5, 0x7BFF = 65504, 0x7C00 / 0xFC00 = +-inf, 0x7E00 NaN
    assert amax(u([0xBC00, 0x4500]), F16, 0, 2) == 5.0
    assert amax(u([0x7BFF, 0xFBFF]), F16, 0, 2) == 65504.0
    assert amax(u([0x0001]), F16, 0, 1) == 2.0 ** -24
    assert amax(u([0xFC00, 0x0000]), F16, 0, 2) == math.inf
    assert math.isnan(amax(u([0x7C00, 0x7E00]), F16, 0, 2))


def test_grad_check_constant_replicas_fill_every_read_bucket():
    """Replica q holding the constant -(q + 1) everywhere: every bucket the
    step reads shows q + 1 for replica q; a bucket holding none of the
    selected rank's elements shows 0."""
    params = [dict(numel=n, dtype=d)
              for n, d in [(700, BF16), (5, F32), (1300, BF16), (33, F32), (90, BF16), (450, BF16)]]
    m = oracle.ShardMap(params, 4, 400, True)
    empty_seen = False
    for ranks in ([0, 1, 2, 3], [2], [3]):
        grads, st, pb = [], [], []
        for bi, buf in enumerate(m.buffers):
            grads.append([np.full(buf.numel, -(q + 1.0), np.float32) for q in range(4)])
            n_local = len(ranks) * m.shard_numel(bi)
            st.append({"exp_avg": np.zeros(n_local, np.float32), "exp_avg_sq": np.zeros(n_local, np.float32),
                       **({"master": np.zeros(n_local, np.float32)} if buf.param_dtype != F32 else {})})
            pb.append(np.zeros(buf.numel, np.uint16 if buf.param_dtype != F32 else np.float32))
        res = oracle.step(m, ranks, grads, st, pb, W.HP, 1, check_grads=True)
        amax = res["grad_amax"]
        total = sum(len(b.buckets) for b in m.buffers)
        assert amax.shape == (4, total) and total == 4
        col = 0
        for bi, buf in enumerate(m.buffers):
            for b, bucket in enumerate(buf.buckets):
                read = any(m.rank_views(bi, b, r) for r in ranks)
                empty_seen |= not read
                for q in range(4):
                    assert amax[q, col] == ((q + 1.0) if read else 0.0), (ranks, bi, b, q)
                col += 1
    assert empty_seen  # rank 3's slice of the fp32 bucket is all padding

def test_grad_check_locates_each_planted_value():
    """Brute force over a tiny two-buffer map with padding: a large value
    planted at one element of one replica shows up at exactly (that replica,
    the element's bucket) when the element belongs to a param of a selected
    rank's shard, and nowhere when it sits in padding or in another rank's
    shard.  The element's bucket is found here from the bucket offsets."""
    params = [dict(numel=n, dtype=d) for n, d in [(70, BF16), (5, F32), (130, BF16), (33, F32)]]
    m = oracle.ShardMap(params, 4, 100, True)
    base = 0.25
    offsets = [0]
    for buf in m.buffers:
        offsets.append(offsets[-1] + len(buf.buckets))
    for ranks in ([0, 1, 2, 3], [1]):
        for bi, buf in enumerate(m.buffers):
            owned = np.zeros(buf.numel, bool)
            for pid in buf.params:
                s0, e0, _ = buf.index[pid]
                owned[s0:e0] = True
            for w in range(0, buf.numel, 3):
                b = next(k for k, bk in enumerate(buf.buckets) if bk.offset <= w < bk.offset + bk.numel)
                slice_rank = (w - buf.buckets[b].offset) // (buf.buckets[b].numel // 4)
                seen = bool(owned[w]) and slice_rank in ranks
                q = w % 4
                grads = [[np.full(bb.numel, base, np.float32) for _ in range(4)] for bb in m.buffers]
                grads[bi][q][w] = -1.0e3
                st = [{"exp_avg": np.zeros(len(ranks) * m.shard_numel(i), np.float32),
                       "exp_avg_sq": np.zeros(len(ranks) * m.shard_numel(i), np.float32),
                       **({"master": np.zeros(len(ranks) * m.shard_numel(i), np.float32)}
                          if bb.param_dtype != F32 else {})} for i, bb in enumerate(m.buffers)]
                pb = [np.zeros(bb.numel, np.uint16 if bb.param_dtype != F32 else np.float32) for bb in m.buffers]
                amax = oracle.step(m, ranks, grads, st, pb, W.HP, 1, check_grads=True)["grad_amax"]
                hit = np.argwhere(amax == 1.0e3)
                if seen:
                    assert hit.tolist() == [[q, offsets[bi] + b]], (ranks, bi, w)
                else:
                    assert len(hit) == 0, (ranks, bi, w)
                assert set(np.unique(amax[amax != 1.0e3])) <= {0.0, base}


def test_grad_check_nan_in_any_piece_makes_the_bucket_nan():
    """A bucket holding several params: a NaN at any element a selected
    rank reads makes that replica's entry NaN, whichever piece it sits in
    and whatever the other pieces hold; the other replicas' entries keep
    their largest magnitude."""
    params = [dict(numel=n, dtype=BF16) for n in (40, 24, 64, 8)]
    m = oracle.ShardMap(params, 2, 10**6, True)
    (buf,) = m.buffers
    assert len(buf.buckets) == 1
    owned = [w for pid in buf.params for w in range(buf.index[pid][0], buf.index[pid][1])]
    assert len(owned) == 136
    for w in owned[::3] + [owned[-1]]:
        q = w % 2
        grads = [[np.full(buf.numel, 2.0, np.float32) for _ in range(2)]]
        grads[0][q][w] = np.nan
        st, pb = _zero_state(m, [0, 1])
        amax = oracle.step(m, [0, 1], grads, st, pb, W.HP, 1, check_grads=True)["grad_amax"]
        assert math.isnan(amax[q, 0]) and amax[1 - q, 0] == 2.0, w


def test_stream_sumsq_equals_array_path():
    n_rep = 8
    keys = [synth.key(3, synth.STREAM_GRAD, 1, k) for k in range(n_rep)]
    for gdt, kind in ((F32, synth.OUT_F32), (BF16, synth.OUT_BF16), (F16, synth.OUT_F16)):
        reps = [synth.normal(5000, k, 1234, 1e-3, kind) for k in keys]
        main, bad = oracle.reduce_prepare(reps, gdt, 0, 5000, 0.5)
        s_arr = float(np.sum(main.astype(np.float64) ** 2))
        s, b = oracle.stream_sumsq(keys, gdt, synth.factor(1e-3), 1234, 5000, 0.5)
        assert bad == b == 0 and abs(s - s_arr) <= 1e-12 * s_arr
        # the streamed main grads themselves, also with two instances and averaging
        for n_inst, avg in ((1, False), (2, True)):
            want, wbad = oracle.reduce_prepare(reps, gdt, 0, 5000, 0.5, n_inst, avg)
            got, gbad = oracle.stream_reduce_prepare(keys, gdt, synth.factor(1e-3), 1234, 5000,
                                                     inv_scale=0.5, n_inst=n_inst, average=avg)
            assert gbad == wbad == 0 and got.tobytes() == want.tobytes()
    # and their count of non-finite main grads: two unit-variance fp32
    # replicas averaged, unscaled by 3e38, overflow wherever the reduced
    # grad exceeds about 1.13 in magnitude
    reps = [synth.normal(5000, k, 77, 1.0) for k in keys[:2]]
    want, wbad = oracle.reduce_prepare(reps, F32, 0, 5000, 3e38)
    got, gbad = oracle.stream_reduce_prepare(keys[:2], F32, synth.factor(1.0), 77, 5000, inv_scale=3e38)
    assert gbad == wbad == int(np.count_nonzero(~np.isfinite(want))) > 0
    assert np.array_equal(np.isfinite(got), np.isfinite(want))


# --------------------------------------------------------------------------
# the seeded generator itself


def test_generator_matches_published_splitmix64():
    g = _golden("splitmix64_seed1234567.json")
    L = synth.host()
    assert [int(L.synth_bits_at(g["seed"], i)) for i in range(5)] == [int(x) for x in g["outputs"]]


def test_generator_truncations_are_exact_16_bit_values():
    k = synth.key(1, synth.STREAM_PARAM, 0, 0)
    v = synth.normal(50000, k, 0, 0.02, synth.OUT_F32_OF_BF16)
    b = synth.normal(50000, k, 0, 0.02, synth.OUT_BF16)
    assert (v.view(np.uint32) >> 16 == b).all()
    v16 = synth.normal(50000, k, 0, 0.02, synth.OUT_F32_OF_F16)
    b16 = synth.normal(50000, k, 0, 0.02, synth.OUT_F16)
    assert (b16.view(np.float16).astype(np.float32) == v16).all()
    x = synth.normal(50000, k, 0, 0.02)
    assert (np.abs(v16) <= np.abs(x)).all() and (np.abs(v) <= np.abs(x)).all()
    assert abs(float(x.std()) - 0.02) < 5e-4


# --------------------------------------------------------------------------
# A7 the fp16 dynamic loss scale


def test_loss_scale_starts_at_the_deepspeed_initial_scale_power():
    g = _golden("deepspeed_fp16_config.json")
    assert g["fp16"]["loss_scale"] == 0  # 0 selects the dynamic scale
    assert oracle.initial_scale(g["fp16"]["initial_scale_power"]) == g["expected_initial_scale"]
    assert oracle.LossScale().scale == g["expected_initial_scale"]
    # a clean step of a fresh scale changes nothing until the growth interval
    s = oracle.LossScale()
    assert s.update(False) == g["expected_initial_scale"]


@pytest.mark.parametrize("growth,backoff,interval,p_inf", [(2.0, 0.5, 1, 0.4), (2.0, 0.5, 3, 0.25),
                                                           (2.0, 0.5, 1000, 0.002), (4.0, 0.25, 2, 0.4)])
def test_loss_scale_hysteresis_1_equals_torch_gradscaler_update(growth, backoff, interval, p_inf):
    """With one hysteresis strike the dynamic scale follows the backoff and
    growth rule of torch's GradScaler (torch._amp_update_scale_, an
    independent library routine) after every step of a seeded inf pattern.
    Powers of two keep both exact; min_scale is set below every scale the
    pattern reaches, since torch has no floor."""
    rng = random.Random(int(growth * 1000 + interval))
    s = oracle.LossScale(2.0**16, growth, backoff, interval, hysteresis=1, min_scale=2.0**-140)
    t_scale = torch.tensor([2.0**16], dtype=torch.float32)
    t_track = torch.tensor([0], dtype=torch.int32)
    steps = 3000 if interval == 1000 else 300
    for step in range(steps):
        found = rng.random() < p_inf
        s.update(found)
        torch._amp_update_scale_(t_scale, t_track, torch.tensor([1.0 if found else 0.0]), growth,
                                 backoff, interval)
        assert s.scale == t_scale.item(), step
        assert 2.0**-126 <= s.scale < 2.0**127


def test_loss_scale_hand_worked_hysteresis_growth_and_floor():
    """Sequences worked by hand from the rule: strikes absorb overflows,
    the last strike backs off, growth restores the strikes, an overflow
    restarts the run of clean steps, and the scale never drops below
    min_scale."""
    s = oracle.LossScale(65536.0, 2.0, 0.5, growth_interval=3, hysteresis=2)
    seq = [(True, 65536.0),    # first strike absorbed
           (True, 32768.0),    # second strike: halve
           (True, 16384.0),    # no strike left: halve again
           (False, 16384.0), (False, 16384.0),
           (True, 8192.0),     # breaks the clean run; still no strike left
           (False, 8192.0), (False, 8192.0),
           (False, 16384.0),   # three clean in a row: grow, strikes back to 2
           (True, 16384.0),    # absorbed again
           (False, 16384.0), (False, 16384.0), (False, 32768.0)]
    for i, (found, want) in enumerate(seq):
        assert s.update(found) == want, i
    f = oracle.LossScale(4.0, 2.0, 0.5, growth_interval=1000, hysteresis=1, min_scale=1.0)
    assert [f.update(True) for _ in range(4)] == [2.0, 1.0, 1.0, 1.0]
    g = oracle.LossScale(1.0, 2.0, 0.5, growth_interval=1, hysteresis=3, min_scale=1.0)
    assert [g.update(False) for _ in range(3)] == [2.0, 4.0, 8.0]
    assert [g.update(True) for _ in range(3)] == [8.0, 8.0, 4.0]
    assert oracle.LossScale(3.0).inv_scale() == float(np.float32(1.0 / 3.0))
