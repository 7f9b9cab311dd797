"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times (same map, layout, rank selection, sizes and entry point),
over every step the workloads configure.

The oracle cannot hold these inputs, so each step it checks:
  - found_inf exactly, and the grad norm against the oracle's own fp64 sum
    of squares streamed from the generator over every element (rel 1e-5);
  - every element of the shard for the bench workload (Llama-7B DP=8) and
    Llama-1.3B fp16 (and for two steps of the 2 x 8 hierarchy at each bucket
    size), and elsewhere a window of whole buckets (at least 64M
    elements: the first, middle and last bucket of the 16-bit buffer, more
    buckets from both ends, and every bucket of the fp32 norm-weight
    buffer), element by element: the oracle redraws the main grads from the
    generator and carries master, m and v from step to step; main grad
    bit-exact, master/m/v within 4 ulp or 1e-6 of the operand scale, 16-bit
    params within 1 ulp;
  - thousands of sampled elements elsewhere -- the first and last element of
    every param piece plus random ones -- recomputed from their replica
    grads at the same tolerances.
A step with an injected inf must leave every sampled and window element
bit-identical.
"""

import math
import os

import numpy as np
import pytest

from synth import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gpu_harness as H  # noqa: E402
import oracle  # noqa: E402

INF_BITS = {H.F32: float("inf"), H.BF16: 0x7F80, H.F16: 0x7C00}
STATE = ("master", "exp_avg", "exp_avg_sq")
# Through the bounds-checked debug build (test_bounds_checked_gpu) each
# workload runs two steps: every step repeats the first one's launches with
# the same geometry, so more steps check no further access.
STEP_CAP = 2 if os.path.basename(os.environ.get("DOPT_LIBRARY") or "") == "libdopt_checked.so" else None


def _inf_position(fc):
    buf = fc.om.buffers[0]
    target = int(buf.numel_unpadded * fc.cfg["inf_at"]["buffer_frac"])
    best = None
    for pid in buf.params:
        s, e, _ = buf.index[pid]
        if e > target and e > s:
            w = max(s, target)
            best = w if best is None else min(best, w)
    return best


def _run(cfg, steps, n_random=3000, window=True, every=False):
    """Steps a workload at full size.  window: compare a window of whole
    buckets element by element (every: the window is the whole shard);
    always: found_inf, the streamed norm and sampled elements."""
    if STEP_CAP is not None:
        steps = min(steps, STEP_CAP)
    fc = H.FullCase(cfg)
    samples = fc.choose_samples(n_random)
    st = fc.initial_sample_state(samples)
    if window:
        if every:
            buckets = [(bi, b) for bi, buf in enumerate(fc.om.buffers) for b in range(len(buf.buckets))]
        else:
            buckets = fc.window_buckets()
        wp = fc.window_pieces(buckets)
        wst = fc.window_initial_state(wp)
        n_win = sum(wst[bi]["master"].size for bi in wst)
        n_pieces = sum(n for *_, n in fc.pieces())
        assert n_win == n_pieces if every else n_win >= min(64 << 20, n_pieces // 2)
    t_applied = 0
    L = oracle.lib()
    for t_step in range(1, steps + 1):
        fc.fill_grads(t_step)
        spec = cfg.get("inf_at")
        inject = spec is not None and spec["step"] == t_step
        if inject:
            assert cfg["layout"] == "full"
            fc.reps[0][spec["replica"]][_inf_position(fc)] = INF_BITS[fc.om.buffers[0].grad_dtype]
        before_dev = fc.device_samples(st)
        before_win = [fc.window_device(sub) for sub, _ in H.window_chunks(wp, wst, 64 << 20)] \
            if (inject and window) else None
        t = t_applied + 1
        found, norm = fc.step(t)
        if inject:
            assert found and math.isnan(norm)
            after = fc.device_samples(st)
            for bi in after:
                for k in STATE + ("param",):
                    assert after[bi][k].tobytes() == before_dev[bi][k].tobytes(), (bi, k)
            if window:
                for (sub, _), bw in zip(H.window_chunks(wp, wst, 64 << 20), before_win):
                    aw = fc.window_device(sub)
                    for bi in aw:
                        for k in STATE + ("param",):
                            assert aw[bi][k].tobytes() == bw[bi][k].tobytes(), (bi, k)
            continue
        sumsq, bad = fc.oracle_sumsq(t_step)
        assert bad == 0 and not found
        o_norm, coef = oracle.ctypes_double(), oracle.ctypes_double()
        clip = L.or_clip_coef(sumsq, cfg["max_norm"], oracle.ctypes_byref(o_norm),
                              oracle.ctypes_byref(coef))
        assert abs(norm - o_norm.value) <= 1e-5 * o_norm.value, (t_step, norm, o_norm.value)
        prev = {bi: {k: v.copy() for k, v in s.items() if k != "sel"} for bi, s in st.items()}
        mains = fc.oracle_samples(st, t_step, t, coef.value, clip)
        got = fc.device_samples(st)
        for bi, s in st.items():
            g = got[bi]
            assert np.array_equal(g["main"].view(np.uint32), mains[bi].view(np.uint32)), (t_step, bi)
            for k in STATE:
                ok = H.state_close(g[k], s[k], prev[bi][k])
                assert ok.all(), (t_step, bi, k, int((~ok).sum()))
            if s["param"].dtype == np.uint16:
                assert H.ulp16(g["param"], s["param"]).max() <= 1, (t_step, bi)
        if window:
            # a group of whole param pieces at a time: oracle, device, compare
            for sub, views in H.window_chunks(wp, wst, 64 << 20):
                wprev = {bi: {k: views[bi][k].copy() for k in STATE} for bi in views}
                res, wbad = fc.window_oracle_step(sub, views, t_step, t, coef.value, clip)
                assert wbad == 0
                want = {bi: dict(views[bi], main=res[bi]["main"], param=res[bi]["param"]) for bi in views}
                findings = H.window_compare(fc.window_device(sub), want, wprev)
                assert not findings, (t_step, findings[:10])
        t_applied += 1
    del fc
    torch.cuda.empty_cache()


def test_bench_workload_llama7b_dp8_rank0():
    # every element of the shard (842,301,952), every configured step; the
    # oracle carries master, m and v of all of them (about 10 GB of host memory)
    cfg = W.config("llama_7b_dp8_rank0")
    _run(cfg, steps=cfg["steps"], every=True)


@pytest.mark.parametrize("size", ["1m", "10m", "40m", "100m"])
def test_hierarchical_llama7b_dp16_2x8(size):
    # 2 instances x 8 ranks, every bucket size of the sweep, all steps
    cfg = W.config("llama_7b_dp16_2x8_" + size)
    _run(cfg, steps=cfg["steps"])
    _run(cfg, steps=2, n_random=0, every=True)  # and the whole shard for two steps


def test_average_in_collective_llama7b_dp8_rank0():
    _run(W.config("llama_7b_dp8_rank0_avg"), steps=1)


def test_dp16_one_instance_general_reduce_kernel():
    # 16 replicas in one instance: the reduce pass's general kernel
    _run(W.config("llama_7b_dp16_rank0"), steps=1)


def test_gpt2_small_all_ranks_with_skipped_step():
    cfg = W.config("gpt2_small_dp8")
    _run(cfg, steps=cfg["steps"])


def test_llama_1p3b_fp16_loss_scaled():
    # every element of all 8 ranks' shards (1,345,423,360), every step
    cfg = W.config("llama_1p3b_fp16_dp8")
    _run(cfg, steps=cfg["steps"], every=True)


def test_bf16_replica_grads_fp32_accumulation():
    _run(W.config("llama_7b_dp8_rank0_bf16grads"), steps=1)


def test_param_larger_than_2_pow_31_elements():
    """One bf16 param of 2^31 + 12345 elements (DP=2, shard-only layout):
    runs are cut at 2^30 elements and every index is 64-bit; the sampled
    elements include both sides of every cut and the ragged end."""
    n = (1 << 31) + 12345
    cfg = W._cfg(name="huge", params=[dict(name="huge", numel=n, dtype=W.BF16),
                                      dict(name="tail", numel=77, dtype=W.F32)],
                 dp=2, bucket_size=None, layout="shard", ranks=[1], steps=1, seed=21)
    _run(cfg, steps=1, n_random=2000, window=False)


def test_grad_check_at_full_size_bench_workload():
    """The pre-reduction grad check on the bench workload, in the launch
    configuration `bench.py --check-grads` times: for the first, a middle
    and the last bucket of the bf16 buffer and the fp32 buffer's bucket, the
    largest |g| of every replica over the rank's pieces, regenerated on the
    host from the seeded generator, equals the device table exactly."""
    import synth
    cfg = W.config("llama_7b_dp8_rank0")
    fc = H.FullCase(cfg)
    fc.fill_grads(1)
    D = H.dopt()
    total = D.dopt_total_buckets(fc.pm)
    amax = torch.full((fc.n_rep, total), -1.0, dtype=torch.float32, device="cuda")
    found, _ = fc.step(1, grad_amax=amax)
    assert not found
    got = amax.cpu().numpy()
    assert (got > 0).all()  # every bucket holds some of rank 0's elements
    r = fc.ranks[0]
    kind = {H.F32: synth.OUT_F32, H.BF16: synth.OUT_BF16, H.F16: synth.OUT_F16}
    checked = 0
    for bi, buf in enumerate(fc.om.buffers):
        nbk = len(buf.buckets)
        for b in sorted({0, nbk // 2, nbk - 1}):
            col = oracle.bucket_number(fc.om, bi, b)
            for k in range(fc.n_rep):
                key = synth.key(fc.seed, synth.STREAM_GRAD, 1, k)
                m = 0.0
                for pid, pb, v in fc.om.rank_pieces(bi, r):
                    if pb != b:
                        continue
                    g = v["gbuf_world"]
                    vals = synth.normal(g.size, key, g.start, cfg["grad_sigma"], kind[buf.grad_dtype])
                    m = max(m, float(np.abs(vals.astype(np.float32)).max()))
                assert got[k, col] == np.float32(m), (bi, b, k, got[k, col], m)
                checked += 1
    assert checked >= 8 * 4
