"""The C ABI from C: tests/c_client/dopt_client.c, a plain C11 program
compiled against include/dopt.h and linked to the library, builds a shard
map and (on a GPU) runs one fused step on cudaMalloc'd buffers.  Its map is
compared with the oracle's shard map, and its step with the oracle's step
on the same inputs (the formulas of the C file, restated here)."""

import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_client", "dopt_client.c")
LIBDIR = os.path.join(ROOT, "mixed_precision_adam_gb300", "lib")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")
F32, BF16 = oracle.F32, oracle.BF16

# the client's fixed problem
PARAMS = [dict(numel=1000, dtype=BF16, wd_mult=1.0), dict(numel=300, dtype=F32, wd_mult=0.0),
          dict(numel=2500, dtype=BF16, wd_mult=1.0), dict(numel=77, dtype=BF16, new_bucket=True, wd_mult=0.5)]
DP, BUCKET = 4, 1500
HP = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
MAX_NORM = 0.5


def _compile(out, cuda):
    if shutil.which("gcc") is None or not os.path.exists(os.path.join(LIBDIR, "libdopt.so")):
        pytest.skip("needs gcc and the built library")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", "-I" + os.path.join(ROOT, "include"), SRC,
           "-o", out]
    if cuda:
        cmd[1:1] = ["-DDOPT_CLIENT_CUDA", "-I" + os.path.join(CUDA, "include")]
        cmd += ["-L" + os.path.join(CUDA, "lib64"), "-lcudart"]
    cmd += ["-L" + LIBDIR, "-ldopt", "-Wl,-rpath," + LIBDIR]
    subprocess.run(cmd, check=True, capture_output=True, text=True)


def test_c_client_shard_map_equals_oracle(tmp_path):
    exe = str(tmp_path / "dopt_client")
    _compile(exe, cuda=False)
    out = subprocess.run([exe, "map"], check=True, capture_output=True, text=True).stdout.splitlines()
    om = oracle.ShardMap(PARAMS, DP, BUCKET, True)
    assert out[0] == f"buffers {len(om.buffers)}"
    want = []
    for bi, buf in enumerate(om.buffers):
        want.append(f"buffer {bi} param_dtype {buf.param_dtype} grad_dtype {buf.grad_dtype} numel {buf.numel} "
                    f"numel_unpadded {buf.numel_unpadded} shard_numel {om.shard_numel(bi)} "
                    f"buckets {len(buf.buckets)}")
        for k, bk in enumerate(buf.buckets):
            want.append(f"bucket {bi} {k} offset {bk.offset} numel {bk.numel} numel_unpadded {bk.numel_unpadded}")
        for r in range(DP):
            for pid, b, v in om.rank_pieces(bi, r):
                want.append(f"piece {bi} {r} param {pid} bucket {b} world {v['gbuf_world'].start} "
                            f"{v['gbuf_world'].end} param_range {v['param'].start} {v['param'].end} "
                            f"shard_offset {v['shard_offset']}")
    assert out[1:] == want


def _grad(b, k, n):
    i = np.arange(n, dtype=np.int64)
    return (((i * 37 + k * 11 + b * 5) % 29 - 14) / 1024.0).astype(np.float32)


def _param(b, n):
    i = np.arange(n, dtype=np.int64)
    return (((i * 13 + b) % 41 - 20) / 256.0).astype(np.float32)


@pytest.mark.gpu
def test_c_client_step_equals_oracle(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import gpu_harness as H
    exe = str(tmp_path / "dopt_client_cuda")
    _compile(exe, cuda=True)
    run = subprocess.run([exe, "step", str(tmp_path)], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, run.stderr
    found, norm = open(tmp_path / "result.txt").read().split()

    om = oracle.ShardMap(PARAMS, DP, BUCKET, True)
    ranks = list(range(DP))
    grads, params, state, masks = [], [], [], []
    for bi, buf in enumerate(om.buffers):
        n, S = buf.numel, om.shard_numel(bi)
        grads.append([_grad(bi, k, n) for k in range(DP)])
        p = _param(bi, n)
        params.append(p.view(np.uint32).__rshift__(16).astype(np.uint16) if buf.param_dtype == BF16 else p.copy())
        st = {"exp_avg": np.zeros(DP * S, np.float32), "exp_avg_sq": np.zeros(DP * S, np.float32)}
        mask = np.zeros(DP * S, bool)
        master = np.zeros(DP * S, np.float32)
        for r in ranks:
            for _, _, v in om.rank_pieces(bi, r):
                lo, w = r * S + v["shard_offset"], v["gbuf_world"]
                master[lo:lo + w.size] = p[w.start:w.end]
                mask[lo:lo + w.size] = True
        if buf.param_dtype != F32:
            st["master"] = master
        state.append(st)
        masks.append(mask)
    before = [{k: v.copy() for k, v in st.items()} for st in state]
    res = oracle.step(om, ranks, grads, state, params, HP, 1, max_norm=MAX_NORM)

    assert int(found) == int(res["found_inf"]) == 0
    assert abs(float(norm) - res["norm"]) <= 1e-5 * res["norm"]
    for bi, buf in enumerate(om.buffers):
        mask = masks[bi]
        for name in ("exp_avg", "exp_avg_sq", "master"):
            if name not in state[bi]:
                continue
            got = np.fromfile(tmp_path / f"b{bi}_{name}.bin", dtype=np.float32)
            assert H.state_close(got[mask], state[bi][name][mask], before[bi][name][mask]).all(), (bi, name)
        if buf.param_dtype == BF16:
            got = np.fromfile(tmp_path / f"b{bi}_param.bin", dtype=np.uint16)
            assert H.ulp16(got, params[bi]).max() <= 1, bi
        else:
            got = np.fromfile(tmp_path / f"b{bi}_param.bin", dtype=np.float32)
            p0 = _param(bi, buf.numel)
            assert H.state_close(got, params[bi], p0).all(), bi
