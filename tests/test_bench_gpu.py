"""The benchmark's GPU modes run and print the lines the contract and the
design notes rely on, on small cases: the main line (with its roofline,
e2e, launches and clocks), the graph-replay comparison and the
bucket-staged comparison."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*argv):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *argv], cwd=ROOT,
                         capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


def test_main_line_on_a_small_case():
    d = _bench("--layers", "2", "--steps", "5", "--warmup", "3", "--e2e-steps", "2",
               "--no-cpu-baseline", "--other-configs", "toy_mlp_dp4")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks", "read_once_ideal"):
        assert key in d, key
    assert d["steps"] == 5 and d["warmup"] == 3 and d["value"] > 0
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["achieved"] > 0 and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    # two buffers (bf16 and fp32 norms): two reduce and two AdamW launches a step
    assert d["gpu_launches"] == 4 * 5
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert e["value"] < d["value"]  # the host copies are inside the end-to-end time
    # one more workload, timed the same way after the main one
    (o,) = d["other_configs"]
    assert "error" not in o, o
    assert o["workload"] == "toy_mlp_dp4" and o["value"] > 0 and o["ms_per_step"] > 0
    assert 0 < o["hbm_frac"] and 0 < o["reduce_prepare_frac"] and 0 < o["adamw_frac"]
    assert o["gpu_launches"] == 2 * o["steps"]  # one reduce and one AdamW launch a step
    assert o["config"]["workload"].startswith("toy_mlp_dp4:")


def test_graph_replay_line():
    d = _bench("--graph", "--workload", "toy_mlp_dp4", "--steps", "20", "--warmup", "3")
    for key in ("dopt_step_ms", "dopt_step_async_ms", "graph_replay_ms"):
        assert d[key] > 0, key


def test_bucket_staged_line():
    d = _bench("--staged", "--layers", "2", "--steps", "5", "--warmup", "3")
    assert d["buckets"] > 1
    assert d["produce_then_fused_ms"] > 0 and d["bucket_staged_overlapped_ms"] > 0


def test_multirank_line():
    d = _bench("--multirank", "--layers", "2", "--steps", "5", "--warmup", "3")
    for key in ("host_combined_ms", "device_combined_ms", "device_graph_ms"):
        assert d[key] > 0, key
