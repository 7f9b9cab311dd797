"""The benchmark's reference arm (the CPU oracle on a bounded sample) runs
without a GPU: its one JSON line must carry the keys the benchmark contract
names, with the reference arm's own e2e and cpu_baseline entries."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "toy_mlp_dp4", "--steps", "2", "--warmup", "1"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "impl",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1
    assert d["value"] > 0 and d["higher_is_better"] is True and d["vs_baseline"] is None
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_recorded_traffic_applies_only_to_the_captured_variant():
    """The committed DRAM-traffic record scales to a launch of the kernel
    variant it was captured on, and to no other (another replica count,
    dtype, layout, averaging or grad check moves other bytes)."""
    sys.path.insert(0, ROOT)
    import bench
    from synth import workloads as W
    rec = json.load(open(os.path.join(ROOT, "profiles", "ncu_k1_traffic.json")))
    default = bench.k1_variant(W.config("llama_7b_dp8_rank0"), False)
    assert rec["variant"] == default
    got = bench.recorded_traffic(1000, default)
    if bench.k1_source_sha256() == rec["source_sha256"]:
        assert got == rec["dram_bytes_per_element"] * 1000
    else:
        assert got is None
    for name, check in (("toy_mlp_dp4", False), ("llama_7b_dp8_rank0_bf16grads", False),
                        ("llama_7b_dp8_rank0_avg", False), ("llama_7b_dp16_2x8_40m", False),
                        ("llama_7b_dp8_rank0", True)):
        assert bench.recorded_traffic(1000, bench.k1_variant(W.config(name), check)) is None, name


def test_clock_records_that_are_rejected():
    """A timed region is taken again when a hardware or thermal slowdown was
    active, or when SM clocks sat well below their maximum with no reason
    (a clock lock); a power cap alone is kept."""
    sys.path.insert(0, ROOT)
    import bench
    ok = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 10}
    assert not bench.clocks_rejected(ok)
    assert not bench.clocks_rejected(dict(ok, sm_mhz=1600.0, reasons=["sw_power_cap"]))
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert bench.clocks_rejected(dict(ok, reasons=[r]))
    assert bench.clocks_rejected(dict(ok, sm_mhz=1200.0))
    assert not bench.clocks_rejected(dict(ok, sm_mhz=None, sm_max_mhz=None, samples=0))
    assert bench.any_rank(True, 1) and not bench.any_rank(False, 1)


def test_both_arms_count_the_same_workload():
    """The reference arm counts the stepped elements with the oracle's shard
    map, the GPU arm with the library's: the two agree on every workload, so
    both lines carry the same config."""
    sys.path.insert(0, ROOT)
    import bench
    import mixed_precision_adam_gb300 as D
    from synth import workloads as W
    for name in W.NAMES:
        cfg = W.config(name)
        pm = D.dopt_build_shard_map(cfg["params"], cfg["dp"], cfg["bucket_size"],
                                    cfg["grad_reduce_in_fp32"], False)
        ranks = list(range(cfg["dp"])) if cfg["ranks"] == "all" else list(cfg["ranks"])
        _, _, elements = bench.algorithmic_bytes(D, pm, cfg["dp"] * cfg["n_inst"], ranks)
        assert bench.oracle_counts(cfg)[0] == elements, name


def test_read_once_ideal_is_4n_plus_26_bytes():
    """The read-once ideal of a bf16-param buffer is 4N + 26 B per element
    for N fp32 replicas (2N + 26 for 16-bit grads); an fp32-param buffer
    writes no separate param (4N + 24)."""
    sys.path.insert(0, ROOT)
    import bench
    import mixed_precision_adam_gb300 as D
    for grad_fp32, dp, want in ((True, 8, 4 * 8 + 26), (False, 8, 2 * 8 + 26), (True, 4, 4 * 4 + 26)):
        pm = D.dopt_build_shard_map([dict(numel=1 << 16, dtype=D.BF16)], dp, 0, grad_fp32, False)
        assert bench.read_once_bytes(D, pm, dp, list(range(dp))) == want * (1 << 16)
    pm = D.dopt_build_shard_map([dict(numel=4096, dtype=D.F32)], 4, 0, True, False)
    assert bench.read_once_bytes(D, pm, 4, [1]) == (4 * 4 + 24) * 1024


def test_other_configs_default_and_failure_entry():
    """The default line times the four other workloads; a workload that
    cannot be timed gives an entry with its error instead of raising, so the
    main line still prints."""
    sys.path.insert(0, ROOT)
    import bench
    from synth import workloads as W
    names = bench.parse_args([]).other_configs.split(",")
    assert len(names) == 4 and bench.DEFAULT_WORKLOAD not in names
    assert all(n in W.NAMES for n in names)
    assert bench.parse_args(["--other-configs", ""]).other_configs == ""
    out = bench.other_config("no_such_workload", bench.parse_args([]), 0)
    assert out["workload"] == "no_such_workload" and "KeyError" in out["error"]
