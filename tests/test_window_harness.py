"""The full-size tests' window check, run on the CPU against the array oracle.

The full-size GPU tests recompute a window of whole buckets by redrawing its
replica grads from the generator and stepping per param piece
(FullCase.window_*).  Here that streaming path runs on scaled-down workloads
next to oracle.step on the whole shard, over several steps: every window
element's main grad, master, m, v and param must be bit-identical, so the
window's indexing (rank slots, bucket bases, buffer offsets, weight-decay
groups) is right before it is used to check the GPU.  No GPU is involved.
"""

import numpy as np
import pytest

import gpu_harness as H
import synth
from synth import workloads as W


def _window_case(hc):
    """A FullCase holding only what the window methods read (no device)."""
    fc = object.__new__(H.FullCase)
    fc.cfg, fc.om, fc.ranks = hc.cfg, hc.om, hc.ranks
    fc.n_rep, fc.seed = hc.n_rep, hc.seed
    fc.pkey = synth.key(hc.seed, synth.STREAM_PARAM, 0, 0)
    return fc


@pytest.mark.parametrize("name,min_elems", [("llama_7b_dp8_rank0", 40_000),
                                            ("llama_7b_dp16_2x8_1m", 30_000),
                                            ("llama_1p3b_fp16_dp8", 200_000),
                                            ("gpt2_small_dp8", 1)])
def test_window_equals_array_oracle(name, min_elems):
    cfg = W.mini(name)
    cfg = dict(cfg, inf_at=None, hp=dict(cfg["hp"], weight_decay=0.1))
    if name == "llama_7b_dp8_rank0":  # two weight-decay groups
        cfg["params"] = [dict(p, wd_mult=0.0 if i % 3 == 0 else 1.0) for i, p in enumerate(cfg["params"])]
    hc = H.HostCase(cfg)
    fc = _window_case(hc)
    buckets = fc.window_buckets(min_elems)
    nbk = len(hc.om.buffers[0].buckets)
    assert {(0, 0), (0, nbk - 1)} <= set(buckets)
    assert all((bi, b) in buckets for bi in range(1, len(hc.om.buffers))
               for b in range(len(hc.om.buffers[bi].buckets)))
    wp = fc.window_pieces(buckets)
    wst = fc.window_initial_state(wp)
    for bi, lst in wp.items():
        for pid, lo, w, k, off in lst:
            if "master" in hc.state[bi]:
                want = hc.state[bi]["master"][lo:lo + k]
            else:
                want = hc.params[bi][w:w + k]
            assert wst[bi]["master"][off:off + k].tobytes() == want.tobytes()
    for t_step in (1, 2, 3):
        grads = hc.grads(t_step)
        ores = hc.oracle_step(grads, t_step)
        assert not ores["found_inf"]
        res, bad = fc.window_oracle_step(wp, wst, t_step, t_step, ores["coef"], ores["clip"],
                                         chunk=1000)
        assert bad == 0
        for bi, lst in wp.items():
            st = hc.state[bi]
            for pid, lo, w, k, off in lst:
                sl = slice(off, off + k)
                assert res[bi]["main"][sl].tobytes() == ores["main"][bi][lo:lo + k].tobytes()
                for key in ("exp_avg", "exp_avg_sq"):
                    assert wst[bi][key][sl].tobytes() == st[key][lo:lo + k].tobytes()
                if "master" in st:
                    assert wst[bi]["master"][sl].tobytes() == st["master"][lo:lo + k].tobytes()
                assert res[bi]["param"][sl].tobytes() == hc.params[bi][w:w + k].tobytes()


def test_window_compare_flags_each_kind_of_difference():
    n = 1000
    rng = np.random.RandomState(0)
    base = {"main": rng.randn(n).astype(np.float32), "master": rng.randn(n).astype(np.float32),
            "exp_avg": rng.randn(n).astype(np.float32), "exp_avg_sq": rng.rand(n).astype(np.float32),
            "param": rng.randint(0, 0x7F00, n).astype(np.uint16)}
    prev = {0: {k: base[k].copy() for k in ("master", "exp_avg", "exp_avg_sq")}}
    assert H.window_compare({0: base}, {0: {k: v.copy() for k, v in base.items()}}, prev, chunk=256) == []
    for key, bump in (("main", lambda a: np.nextafter(a, np.float32(np.inf))),
                      ("master", lambda a: a * np.float32(1.001)),
                      ("param", lambda a: a + np.uint16(2))):
        got = {k: v.copy() for k, v in base.items()}
        got[key][777] = bump(got[key][777:778])[0]
        found = H.window_compare({0: got}, {0: base}, prev, chunk=256)
        assert len(found) == 1 and key in found[0] and "[768, 1000)" in found[0], found
