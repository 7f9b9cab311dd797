"""Parity of the CUDA path with the CPU oracle, element by element, through
the library's C ABI.  Sizes span many tiles and ragged run ends; the edge
cases cover padding, unaligned runs, every dtype pair, hierarchical DP,
skipped steps and the unclipped branch."""

import copy

import numpy as np
import pytest

from synth import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gpu_harness as H  # noqa: E402


def _check(cfg, steps=None, separate=False):
    ok, report = H.run_parity(cfg, steps, separate)
    assert ok, "\n".join(report)


@pytest.mark.parametrize("name", ["toy_mlp_dp4", "gpt2_small_dp8", "llama_1p3b_fp16_dp8",
                                  "llama_7b_dp8_rank0", "llama_7b_dp16_2x8_1m"])
def test_workload_mini(name):
    _check(W.mini(name))


def test_separate_entry_points_match_oracle():
    _check(W.mini("gpt2_small_dp8"), separate=True)


def _tiny(params, dp, **kw):
    cfg = W._cfg(name="tiny", params=params, dp=dp, steps=3, seed=kw.pop("seed", 7))
    cfg.update(kw)
    return cfg


RAGGED = [dict(numel=n, dtype=d) for n, d in
          [(1, 1), (63, 1), (65, 1), (1000, 0), (127, 1), (4099, 1), (3, 0), (20001, 1), (129, 2)]]


@pytest.mark.parametrize("dp", [1, 3, 8])
@pytest.mark.parametrize("grad_fp32", [True, False])
def test_ragged_params_all_dtypes(dp, grad_fp32):
    _check(_tiny(RAGGED, dp, bucket_size=5000, grad_reduce_in_fp32=grad_fp32,
                 grad_sigma=1e-2, max_norm=0.5))


def test_unaligned_runs_large_dp():
    # DP=32: lcm(32,128)=128, so a 128-element bucket gives 4-element slices
    # that start off the 8-element vector grid
    params = [dict(numel=n, dtype=1) for n in (100, 37, 300, 5, 77)]
    _check(_tiny(params, 32, bucket_size=64))


def test_busbw_padding_and_new_bucket():
    params = [dict(numel=n, dtype=1, new_bucket=(i % 3 == 1)) for i, n in
              enumerate([700, 5000, 33, 12000, 999, 64, 65])]
    _check(_tiny(params, 4, bucket_size=3000, pad_for_high_busbw=True))


def test_weight_decay_multipliers():
    params = [dict(numel=n, dtype=1, wd_mult=w) for n, w in
              [(5000, 1.0), (5000, 0.0), (333, 0.5), (4096, 0.0), (70, 1.0)]]
    _check(_tiny(params, 2, bucket_size=None, warm_state=True))


def test_many_runs_chunked_launches():
    # more runs than one kernel-parameter table holds: alternate wd_mult so
    # neighbouring params never merge into one run
    params = [dict(numel=64 + (i % 5), dtype=1, wd_mult=float(i % 2)) for i in range(2500)]
    _check(_tiny(params, 1, bucket_size=None, steps=2))


@pytest.mark.parametrize("n_runs", [31, 32, 33])
@pytest.mark.parametrize("grad_fp32", [True, False])
def test_run_table_capacity_boundary(n_runs, grad_fp32):
    # a launch of at most 32 runs takes the kernels built for a 32-entry
    # parameter table (the short-launch reduce with fp32 grads, the AdamW
    # pass), a longer one the full table: one rank and one bucket, with
    # alternating wd_mult so that every param is a run of its own
    params = [dict(numel=1000 + 37 * i, dtype=1, wd_mult=float(i % 2)) for i in range(n_runs)]
    _check(_tiny(params, 1, bucket_size=None, grad_reduce_in_fp32=grad_fp32, grad_sigma=1e-2))


@pytest.mark.parametrize("name", ["llama_7b_dp8_rank0", "toy_mlp_dp4"])
def test_state_rewritten_just_before_a_fused_step(name):
    # a kernel that rewrites master (or the fp32 params), m and v is queued
    # right before each fused step on the same stream, with no host
    # synchronisation, and the step must read the new values: the AdamW
    # pass loads its first tile's state ahead of its wait for the reduce
    # pass, which stream order makes safe (the rewriting kernel ends before
    # the reduce pass starts)
    D = H.dopt()
    cfg = W.mini(name)
    hc = H.HostCase(cfg)
    dc = H.DeviceCase(hc)
    report = []
    for t_step in (1, 2, 3):
        grads = hc.grads(t_step)
        t = hc.t_applied + 1
        reps = [[dc._up(r) for r in g] for g in grads]
        torch.cuda.synchronize()
        if t_step > 1:  # exact rewrites: halving, quartering, negation
            for b, st in enumerate(hc.state):
                st["exp_avg"] *= np.float32(0.5)
                dc.exp_avg[b].mul_(0.5)
                st["exp_avg_sq"] *= np.float32(0.25)
                dc.exp_avg_sq[b].mul_(0.25)
                if "master" in st:
                    st["master"] *= np.float32(-1.0)
                    dc.master[b].mul_(-1.0)
                else:
                    hc.params[b] *= np.float32(-1.0)
                    dc.params[b].mul_(-1.0)
        before = H.snapshot(hc)
        ores = hc.oracle_step(grads, t)
        found, norm = D.dopt_step(dc.step_args(reps, t))
        assert H.compare_step(hc, dc, ores, found, norm, before, report), "\n".join(report)
        assert not found
        hc.t_applied += 1


def test_average_in_collective_and_hierarchy():
    params = W.llama(1, 128, 344, 257)
    _check(_tiny(params, 4, bucket_size=20000, average=True, steps=2))
    _check(_tiny(params, 4, bucket_size=20000, n_inst=2, steps=2))
    _check(_tiny(params, 4, bucket_size=20000, n_inst=3, average=True, steps=2,
                 layout="shard", ranks=[2]))


def test_shard_layout_every_rank():
    params = W.llama(1, 96, 256, 131)
    for r in range(4):
        _check(_tiny(params, 4, bucket_size=9000, layout="shard", ranks=[r], steps=2))


@pytest.mark.parametrize("max_norm", [0.0, -1.0, 1e9])
def test_unclipped_branch(max_norm):
    _check(_tiny(RAGGED, 2, bucket_size=5000, max_norm=max_norm))


def test_remote_terms():
    _check(_tiny(RAGGED, 2, bucket_size=5000, remote_sumsq=3.0, steps=2))
    _check(_tiny(RAGGED, 2, bucket_size=5000, remote_found_inf=True, steps=1))


@pytest.mark.parametrize("where", ["first", "last", "fp32_group", "nan"])
def test_nonfinite_skips_step_untouched(where):
    cfg = _tiny(RAGGED, 4, bucket_size=5000, warm_state=True, steps=1)
    hc = H.HostCase(cfg)
    dc = H.DeviceCase(hc)
    grads = hc.grads(1)
    bi = 1 if where == "fp32_group" else 0
    pieces = hc.om.rank_pieces(bi, 3 if where == "last" else 0)
    w = pieces[-1][2]["gbuf_world"].end - 1 if where == "last" else pieces[0][2]["gbuf_world"].start
    val = np.nan if where == "nan" else np.inf
    rep = grads[bi][2]
    if rep.dtype == np.uint16:
        rep[w] = 0x7FC0 if where == "nan" else 0x7F80
    else:
        rep[w] = val
    before = dc.download()
    found, norm = dc.step(grads, 1)
    after = dc.download()
    assert found and np.isnan(norm)
    for b_list, a_list in zip(before[:4], after[:4]):  # params, master, m, v
        for b, a in zip(b_list, a_list):
            if b is not None:
                assert b.tobytes() == a.tobytes()


def test_zero_element_rank():
    # a 10-element param with DP=8: ranks 1..7 own only padding of the
    # 128-element bucket
    params = [dict(numel=10, dtype=1), dict(numel=300, dtype=0)]
    _check(_tiny(params, 8, bucket_size=None, steps=2))
    _check(_tiny(params, 8, bucket_size=None, steps=2, layout="shard", ranks=[5]))


def test_repeat_is_deterministic():
    cfg = W.mini("llama_7b_dp8_rank0")
    outs = []
    for _ in range(2):
        hc = H.HostCase(cfg)
        dc = H.DeviceCase(hc)
        norms = [dc.step(hc.grads(t), t)[1] for t in (1, 2)]
        outs.append((norms, [a.tobytes() for a in dc.download()[1] if a is not None]))
    assert outs[0] == outs[1]


@pytest.mark.parametrize("grad_fp32", [True, False])
def test_scale_gradients_and_zero_count(grad_fp32):
    """scale_gradients(1/num_tokens) with a factor that rounds (1/3), and
    main grads that are exactly zero (zero in every replica) for count_zeros."""
    cfg = _tiny(RAGGED, 4, bucket_size=5000, grad_reduce_in_fp32=grad_fp32, grad_scale=1.0 / 3.0,
                grad_sigma=1e-2, steps=2)
    hc = H.HostCase(cfg)
    dc = H.DeviceCase(hc)
    report = []
    for t in (1, 2):
        grads = hc.grads(t)
        for bi, reps in enumerate(grads):
            for r in reps:
                r[3::97] = 0  # the same positions in every replica
        before = H.snapshot(hc)
        ores = hc.oracle_step(grads, t)
        assert ores["num_zeros"] > 0
        found, norm = dc.step(grads, t)
        assert H.compare_step(hc, dc, ores, found, norm, before, report), "\n".join(report)
        hc.t_applied += 1


def test_dynamic_loss_scaler_through_a_skipped_step():
    """fp16 with a dynamic loss scale through an overflow: the oracle keeps
    its own scale (oracle.LossScale) and steps with it; the device steps
    with the library's scaler (dopt_loss_scaler_*), each side's unscale
    factor from its own scale.  An overflow at step 2 skips the step and
    halves the scale; two clean steps later it grows back.  The two scale
    trajectories must be equal, and so must every step's results."""
    import oracle
    D = H.dopt()
    cfg = W.mini("llama_1p3b_fp16_dp8")
    cfg = dict(cfg, inf_at=dict(step=2, replica=3, buffer_frac=0.3), steps=5)
    hc = H.HostCase(cfg)
    dc = H.DeviceCase(hc)
    o_scale = oracle.LossScale(oracle.initial_scale(16), 2.0, 0.5, growth_interval=2, hysteresis=1)
    scaler = D.dopt_loss_scaler_init(65536.0, 2.0, 0.5, growth_interval=2, hysteresis=1)
    report = []
    o_traj, d_traj = [], []
    for step in range(1, 6):
        o_traj.append(o_scale.scale)
        d_traj.append(scaler.scale)
        grads = hc.grads(step)
        t = hc.t_applied + 1
        before = H.snapshot(hc)
        hc.cfg["loss_scale"] = o_scale.scale  # the oracle's unscale factor
        ores = hc.oracle_step(grads, t)
        hc.cfg["loss_scale"] = scaler.scale  # the device's
        found, norm = dc.step(grads, t)
        hc.cfg["loss_scale"] = o_scale.scale  # compare_step decodes with the oracle's
        assert H.compare_step(hc, dc, ores, found, norm, before, report), "\n".join(report)
        assert found == (step == 2)
        if not found:
            hc.t_applied += 1
        o_scale.update(ores["found_inf"])
        D.dopt_loss_scaler_update(scaler, found)
    assert d_traj == o_traj
    assert o_traj == [65536.0, 65536.0, 32768.0, 32768.0, 65536.0]
    assert scaler.scale == o_scale.scale == 65536.0


def test_bounded_wait_runs_out_and_reports():
    """A tile whose copy is never issued (test hook): the TMA-staged reduce
    gives up after its bounded wait, the step is skipped and reported as a
    kernel error, the state is untouched, and the next step is correct.
    The hook exists in the bounds-checked debug build only, through which
    test_bounds_checked_gpu runs this file again."""
    D = H.dopt()
    if "dopt_debug_starve_copy" not in D.exported_symbols():
        pytest.skip("the copy-starving hook is compiled into the bounds-checked debug build only")
    # enough tiles that the reduce pass takes the bulk-copy kernel
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    params = _tma_sized_params(int(1.25 * 16 * 2048 * sms)) + [dict(numel=4096, dtype=1)]
    cfg = _tiny(params, 2, bucket_size=None, steps=2)
    hc = H.HostCase(cfg)
    dc = H.DeviceCase(hc)
    grads = hc.grads(1)
    before = dc.download()
    D.dopt_debug_starve_copy(0)
    try:
        with pytest.raises(D.DoptError) as e:
            dc.step(grads, 1)
    finally:
        D.dopt_debug_starve_copy(-1)
    assert e.value.status == D.E_CUDA and "gave up waiting" in str(e.value)
    stats = D.dopt_read_step_stats(dc.ws)
    assert stats["kernel_error"] == 1 and stats["found_inf"] == 1
    after = dc.download()
    for b_list, a_list in zip(before[:4], after[:4]):
        for b, a in zip(b_list, a_list):
            if b is not None:
                assert b.tobytes() == a.tobytes()
    # the context is usable and the next step matches the oracle
    report = []
    snap = H.snapshot(hc)
    ores = hc.oracle_step(grads, 1)
    found, norm = dc.step(grads, 1)
    assert H.compare_step(hc, dc, ores, found, norm, snap, report), "\n".join(report)
    assert D.dopt_read_step_stats(dc.ws)["kernel_error"] == 0


@pytest.mark.parametrize("t", [2, 37, 1000, 123_457, 2**31 + 5])
@pytest.mark.parametrize("device_step", [False, True])
def test_bias_correction_at_large_step_numbers(t, device_step):
    """The bias corrections 1 - beta1^t and sqrt(1 - beta2^t) at step
    numbers far past those the workloads reach, where beta^t falls below an
    fp32 ulp of 1: one step from a warm state (nonzero m and v) with step
    number t, from host-computed step scalars and from the device step
    counter (holding t - 1), against the oracle."""
    D = H.dopt()
    cfg = _tiny(RAGGED[:6], 4, bucket_size=3000, warm_state=True, steps=1, grad_sigma=1e-2)
    hc = H.HostCase(cfg)
    dc = H.DeviceCase(hc)
    grads = hc.grads(1)
    before = H.snapshot(hc)
    ores = hc.oracle_step(grads, t)
    if device_step:
        args = dc.step_args([[dc._up(r) for r in g] for g in grads], 1)
        d_step = torch.tensor([t - 1], dtype=torch.int64, device="cuda")
        args.set_device_step(d_step)
        found, norm = D.dopt_step(args)
        assert int(d_step.item()) == (t - 1 if found else t)
    else:
        found, norm = dc.step(grads, t)
    report = []
    assert H.compare_step(hc, dc, ores, found, norm, before, report), "\n".join(report)


def _bf16_value(x):
    """The nearest bf16 value of x, as a float (exact in the bf16 bits)."""
    return float(torch.tensor([x], dtype=torch.float32).to(torch.bfloat16).float().item())


@pytest.mark.parametrize("grad_fp32", [False, True])
@pytest.mark.parametrize("values", ["below_2_62", "above_2_62", "mixed_max"])
def test_huge_finite_grads_are_finite(grad_fp32, values):
    """Finite grads whose squares overflow fp32 (or come within a factor 16
    of it: the largest values the norm's fp32 accumulator takes, 16 of them
    per thread and tile in the 16-bit reduce kernel) must neither set
    found_inf nor lose the norm: every replica holds the same value v at an
    element, so the reduced grad is v exactly, with alternating signs and,
    for "mixed_max", values up to the dtype's largest."""
    big = 2.0**62 * (1 - 2.0**-8)  # bf16-representable, square just below 2^124
    pool = {"below_2_62": [big],
            "above_2_62": [2.0**70, 2.0**100],
            "mixed_max": [big, 2.0**64, 2.0**120, 1.0e-3]}[values]
    pool = [_bf16_value(v) for v in pool]
    cfg = _tiny(RAGGED, 4, bucket_size=5000, grad_reduce_in_fp32=grad_fp32, steps=1, max_norm=1.0)
    hc = H.HostCase(cfg)
    dc = H.DeviceCase(hc)
    grads = hc.grads(1)
    for bi, reps in enumerate(grads):
        n = reps[0].size
        idx = np.arange(n)
        vals = np.array(pool)[idx % len(pool)] * np.where(idx % 2 == 0, 1.0, -1.0)
        if reps[0].dtype == np.uint16:  # a 16-bit grad buffer
            kind = torch.bfloat16 if hc.om.buffers[bi].grad_dtype == H.BF16 else torch.float16
            if kind == torch.float16:  # fp16 grads top out at 65504
                vals = np.clip(vals, -6e4, 6e4)
            bits = torch.from_numpy(vals.astype(np.float32)).to(kind).view(torch.int16).numpy().view(np.uint16)
            for r in reps:
                r[:] = bits
        else:
            for r in reps:
                r[:] = vals.astype(np.float32)
    before = H.snapshot(hc)
    ores = hc.oracle_step(grads, 1)
    assert not ores["found_inf"] and np.isfinite(ores["sumsq"])
    found, norm = dc.step(grads, 1)
    report = []
    assert H.compare_step(hc, dc, ores, found, norm, before, report), "\n".join(report)
    assert not found


@pytest.mark.parametrize("grad_fp32", [False, True])
def test_subnormal_grads_keep_their_values(grad_fp32):
    """Subnormal grads (fp32 and bf16 subnormals, and fp16 subnormals that the
    loss scale divides further) are summed, unscaled and stepped like any
    value on both sides: no flush to zero.  Zeros of both signs mix in."""
    pool = [1.0e-40, -3.0e-39, 1.4e-45, -1.0e-30, 0.0, -0.0, 5.9e-8, -6.0e-8]
    cfg = _tiny(RAGGED, 4, bucket_size=5000, grad_reduce_in_fp32=grad_fp32, steps=1,
                loss_scale=65536.0, max_norm=0.0)
    hc = H.HostCase(cfg)
    dc = H.DeviceCase(hc)
    grads = hc.grads(1)
    for bi, reps in enumerate(grads):
        n = reps[0].size
        vals = np.array(pool, np.float32)[np.arange(n) % len(pool)]
        if reps[0].dtype == np.uint16:
            kind = torch.bfloat16 if hc.om.buffers[bi].grad_dtype == H.BF16 else torch.float16
            bits = torch.from_numpy(vals).to(kind).view(torch.int16).numpy().view(np.uint16)
            for r in reps:
                r[:] = bits
        else:
            for r in reps:
                r[:] = vals
    before = H.snapshot(hc)
    ores = hc.oracle_step(grads, 1)
    assert ores["num_zeros"] > 0 and ores["sumsq"] > 0
    found, norm = dc.step(grads, 1)
    report = []
    assert H.compare_step(hc, dc, ores, found, norm, before, report), "\n".join(report)


@pytest.mark.parametrize("hp", [
    dict(lr=0.0, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1),   # no update at all
    dict(lr=1e-3, beta1=0.0, beta2=0.0, eps=1e-8, weight_decay=0.0),   # m = g, v = g^2
    dict(lr=1e-2, beta1=0.5, beta2=0.999, eps=1.0, weight_decay=1.0),  # eps dominates, strong decay
], ids=["lr0", "beta0", "eps1"])
def test_degenerate_hyperparameters(hp):
    """Edge values the hyper-parameter checks accept, against the oracle over
    three steps from a warm state; with lr = 0 the masters and params stay
    bit for bit what they were."""
    cfg = _tiny(RAGGED, 3, bucket_size=5000, steps=3, warm_state=True, grad_sigma=1e-2, hp=hp)
    _check(cfg)
    if hp["lr"] == 0.0:
        hc = H.HostCase(cfg)
        dc = H.DeviceCase(hc)
        before = [t.clone() for t in dc.params] + [t.clone() for t in dc.master if t is not None]
        for t in range(1, 4):
            found, _ = dc.step(hc.grads(t), t)
            assert not found
        after = list(dc.params) + [t for t in dc.master if t is not None]
        for b, a in zip(before, after):
            assert torch.equal(b, a)


def test_concurrent_steps_from_two_threads_on_two_streams():
    """Two independent optimizers stepped at the same time from two host
    threads, each on its own stream with its own map and workspace: the
    library's per-thread and per-device host state (launch scratch, side
    streams, caches) keeps them apart, and each matches its oracle."""
    import threading
    cfgs = [_tiny(RAGGED, 4, bucket_size=5000, steps=3, seed=31),
            dict(W.mini("llama_7b_dp8_rank0"), steps=3)]
    results = [None, None]

    def run(i):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                hc = H.HostCase(cfgs[i])
                dc = H.DeviceCase(hc)
                report, ok = [], True
                for t_step in range(1, 4):
                    grads = hc.grads(t_step)
                    t = hc.t_applied + 1
                    before = H.snapshot(hc)
                    ores = hc.oracle_step(grads, t)
                    found, norm = dc.step(grads, t)
                    ok &= H.compare_step(hc, dc, ores, found, norm, before, report)
                    if not ores["found_inf"]:
                        hc.t_applied += 1
                s.synchronize()
            results[i] = (ok, report)
        except Exception as e:  # reported below, in the main thread
            results[i] = (False, [repr(e)])

    threads = [threading.Thread(target=run, args=(i,)) for i in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    for ok, report in results:
        assert ok, "\n".join(report)


def test_two_hundred_steps_track_the_oracle():
    """A long run: 200 consecutive steps of a small ragged map with a loss
    scale, a warm start and an inf at step 100 (skipped), every step
    compared with the oracle -- m, v and the masters carry every earlier
    step's rounding, so drift between the two sides would show."""
    cfg = _tiny(RAGGED, 4, bucket_size=5000, steps=200, warm_state=True, grad_sigma=1e-2,
                inf_at=dict(step=100, replica=1, buffer_frac=0.3))
    ok, report = H.run_parity(cfg)
    assert ok, "\n".join(r for r in report if "ok=False" in r or not r.startswith("step"))[:4000]
    assert sum("found_inf=True" in r for r in report) == 1  # the step with the inf, skipped


def _tma_sized_params(scale):
    """Ragged bf16 params (each starts on the 64-element pad, most end off
    the 4- and 8-element grids) totalling `scale` elements or more."""
    sizes = [1_000_003, 777_777, 65, 2_500_001, 999_999, 333, 1_234_567, 4_099, 640_000, 31]
    out, total, i = [], 0, 0
    while total < scale:
        n = sizes[i % len(sizes)]
        out.append(dict(numel=n, dtype=1))
        total += n
        i += 1
    return out


@pytest.mark.parametrize("dp,average,check", [(1, False, False), (2, True, False), (4, False, True),
                                              (8, False, False), (8, True, True)])
def test_tma_staged_reduce_ragged(dp, average, check):
    """fp32 replicas in one instance, every run 8-element aligned, and enough
    tiles (16 x 2048 elements per SM or more) that the reduce pass stages the
    replica tiles through shared memory with bulk copies: ragged run ends
    (the last elements of a run after its last multiple of 4), every
    replica count the staged kernel takes, averaging, and the grad check."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    params = _tma_sized_params(int(1.25 * 16 * 2048 * sms))
    cfg = _tiny(params, dp, bucket_size=3_000_000, grad_reduce_in_fp32=True, average=average, steps=2,
                seed=23 + dp)
    if check:
        ok, report = H.run_check(cfg, [[(0, 0, 3.0)], [(5, dp - 1, -7.5)]])
        assert ok, "\n".join(report)
    else:
        _check(cfg)
