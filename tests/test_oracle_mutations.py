"""The oracle's pins must be able to fail.  Each entry below plants one
plausible mistake (a dropped term, a wrong sign, index or rounding, a
transposed operand, a misread page rule) in a scratch copy of oracle/ and
runs tests/test_oracle_pins.py against that copy: every mutant must fail at
least one pin.  The repository's own oracle is never modified, and a copy of
the unmutated oracle must pass first.  CPU only; the mutants run in parallel.
"""

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C, PY, SM, LS = "oracle/oracle.c", "oracle/__init__.py", "oracle/shard_map.py", "oracle/loss_scale.py"

# (file, text in the oracle, its replacement, what the mistake is)
MUTANTS = [
    # A5 AdamW
    (C, "float bc2_sqrt = (float)sqrt(1.0 - or_pow(hp->beta2, t));", "float bc2_sqrt = 1.0f;",
     "no bias correction of v"),
    (C, "float step_size = (float)(hp->lr / (1.0 - or_pow(hp->beta1, t)));", "float step_size = (float)(hp->lr);",
     "no bias correction of m"),
    (C, "p = p - step_size * (m / denom);", "p = p + step_size * (m / denom);", "update sign"),
    (C, "float v = b2 * exp_avg_sq[j] + (omb2 * g) * g;", "float v = b2 * exp_avg_sq[j] + (omb2 * g);",
     "dropped g factor in v"),
    (C, "float m = b1 * exp_avg[j] + omb1 * g;", "float m = omb1 * exp_avg[j] + b1 * g;", "betas transposed"),
    (C, "float p = master[j] * decay;", "float p = master[j];", "no weight decay"),
    (C, "  float decay = (float)(1.0 - hp->lr * hp->weight_decay * wd_mult);",
     "  float decay = (float)(1.0 - hp->lr * hp->weight_decay);", "wd_mult ignored"),
    (C, "    float denom = sqrtf(v) / bc2_sqrt + eps;", "    float denom = sqrtf(v / bc2_sqrt) + eps;",
     "bias correction inside the square root"),
    (C, "    float denom = sqrtf(v) / bc2_sqrt + eps;", "    float denom = sqrtf(v + eps) / bc2_sqrt;",
     "eps inside the square root"),
    (C, "  float omb1 = (float)(1.0 - hp->beta1), omb2 = (float)(1.0 - hp->beta2);",
     "  float omb1 = 1.0f - b1, omb2 = 1.0f - b2;", "1 - beta from the rounded beta"),
    # A4 norm and clip
    (C, "    coef = max_norm / (norm + 1.0e-6);", "    coef = max_norm / (sumsq + 1.0e-6);", "clip by sumsq"),
    (C, "    coef = max_norm / (norm + 1.0e-6);", "    coef = max_norm / (norm + 1.0e-5);", "clip epsilon"),
    (C, "float g = clip ? main_grad[j] * c : main_grad[j];", "float g = main_grad[j];", "clip not applied"),
    (C, "    clip = coef < 1.0;", "    clip = 1;", "clips when coef >= 1"),
    (C, "  if (max_norm > 0.0) {", "  if (max_norm >= 0.0) {", "max_norm 0 clips"),
    (C, "  for (int64_t j = 0; j < len; ++j) s += (double)main_grad[j] * (double)main_grad[j];",
     "  for (int64_t j = 0; j < len; ++j) s += (double)(main_grad[j] * main_grad[j]);", "squares in fp32"),
    (PY, "    sumsq += remote_sumsq", "    sumsq += 0.0", "remote sum of squares dropped"),
    (PY, "found = bad > 0 or bool(remote_found_inf)", "found = bad > 0", "remote found_inf dropped"),
    # A2 reduce-scatter, A2' scale_gradients, A3 prepare
    (C, "float term = average ? x : x * pre;", "float term = x;", "no prescale"),
    (C, "  float pre = (float)(1.0 / (double)n_rep);", "  float pre = (float)(1.0 / (double)(n_rep / n_inst));",
     "prescale by the instance size"),
    (C, "    s = or_round_to(s, gdt);", "", "no rounding to the grad dtype"),
    (C, "    total = or_round_to(total, gdt);", "", "no rounding after the inter-instance sum"),
    (C, "    if (average) total = total * (float)(1.0 / (double)n_inst);", "", "no inter-instance average"),
    (C, "    if (average) s = s * (float)(1.0 / (double)dpi);", "", "no intra-instance average"),
    (C, "      s = (q == 0) ? term : s + term;", "      s = s + term;", "sum starts from +0"),
    (C, "  return or_round_to(red * factor, gdt);", "  return red * factor;", "scale_gradients not rounded"),
    (C, "  return or_round_to(red * factor, gdt);", "  return red;", "scale_gradients ignored"),
    (C, "float mg = red * inv_scale;", "float mg = red;", "no unscale"),
    (C, "      if (!or_is_finite(mg)) ++bad;", "", "no inf check"),
    (C, "static int or_is_finite(float x) { return (or_f32_bits(x) & 0x7F800000u) != 0x7F800000u; }",
     "static int or_is_finite(float x) { return x == x; }", "infinity counted finite"),
    (PY, "zeros += int(np.count_nonzero(main[local:local + n] == 0))",
     "zeros += int(np.count_nonzero(main[local:local + n]))", "count_zeros counts nonzeros"),
    # the generator-streamed form of A2 + A3 (full-size checks)
    (C, "                                    grad_scale, gdt) * inv_scale;\n      main_out[j] = mg;",
     "                                    grad_scale, gdt);\n      main_out[j] = mg;", "streamed main grads not unscaled"),
    (C, "      main_out[j] = mg;\n      if (!or_is_finite(mg)) ++bad;", "      main_out[j] = mg;",
     "streamed form counts no non-finite main grad"),
    # casts and widening
    (C, "if (rem > 0x8000u || (rem == 0x8000u && (kept & 1u))) kept += 1u;", "if (rem >= 0x8000u) kept += 1u;",
     "bf16 ties away from zero"),
    (C, "    return (uint16_t)(kept | 0x0040u);", "    return (uint16_t)kept;", "bf16 NaN may become inf"),
    (C, "      if (rem > 0x1000u || (rem == 0x1000u && (kept & 1u))) kept += 1u;", "      if (rem >= 0x1000u) kept += 1u;",
     "fp16 ties away from zero"),
    (C, "      if (frac > 0.5f || (frac == 0.5f && (fl & 1u))) fl += 1u;", "      if (frac >= 0.5f) fl += 1u;",
     "fp16 subnormal ties away from zero"),
    (C, "    if (a >= 65520.0f) return", "    if (a > 65504.0f) return", "fp16 overflow threshold"),
    (C, "    float v = ldexpf((float)man, -24);", "    float v = ldexpf((float)man, -23);", "fp16 subnormal scale"),
    (C, "    return or_bits_f32(sign | 0x7F800000u | (man << 13));", "    return or_bits_f32(sign | 0x7F800000u);",
     "fp16 NaN widened to inf"),
    # A2 grad check
    (C, "    if (x != x) return NAN;", "", "grad check: NaN not reported"),
    (C, "    if (x < 0) x = -x;", "", "grad check: no magnitude"),
    (PY, 'return float("nan") if (a != a or b != b) else max(a, b)', "return max(a, b)",
     "grad check: merge drops NaN"),
    (PY, 'return float("nan") if (a != a or b != b) else max(a, b)', 'return float("nan") if (a != a) else max(a, b)',
     "grad check: merge ignores the new run's NaN"),
    (PY, "    return sum(len(buf.buckets) for buf in smap.buffers[:bi]) + b", "    return b",
     "grad check: buckets not numbered across buffers"),
    # step composition
    (PY, 'rep0 = v["gbuf_world"].start if layout == "full" else v["shard_offset"]', 'rep0 = v["gbuf_world"].start',
     "shard-only replicas read at the world index"),
    (PY, 'rep0 = v["gbuf_world"].start if layout == "full" else v["shard_offset"]',
     'rep0 = v["gbuf_world"].start if layout == "full" else v["gbuf_local"].start',
     "shard-only replicas read at the bucket-local index"),
    (PY, '                local = slot * S + v["shard_offset"]', '                local = v["shard_offset"]',
     "rank slot ignored"),
    # A7 loss scale
    (LS, "    return math.ldexp(1.0, int(initial_scale_power))", "    return math.ldexp(1.0, int(initial_scale_power) - 1)",
     "loss scale starts at 2^15"),
    (LS, "                self.scale = max(self.scale * self.backoff_factor, self.min_scale)",
     "                self.scale = max(self.scale, self.min_scale)", "no backoff on an overflow"),
    (LS, "                self.scale = max(self.scale * self.backoff_factor, self.min_scale)",
     "                self.scale = self.scale * self.backoff_factor", "no min_scale floor"),
    (LS, "            if self.strikes_left <= 0:", "            if self.strikes_left < 0:", "one strike too many"),
    (LS, "            self.clean_steps = 0\n            self.strikes_left -= 1",
     "            self.strikes_left -= 1", "an overflow does not restart the clean run"),
    (LS, "                self.strikes_left = self.hysteresis\n", "", "growth does not restore the strikes"),
    (LS, "            if self.clean_steps == self.growth_interval:", "            if self.clean_steps > self.growth_interval:",
     "grows one step late"),
    (LS, "                self.scale = self.scale * self.growth_factor", "                self.scale = self.scale * 2.0",
     "growth factor ignored"),
    # A1 shard map
    (SM, "    for pid in reversed(buf.params):", "    for pid in buf.params:", "forward walk"),
    (SM, "        start = pad_up(cursor, 64)", "        start = cursor", "no 64-element start pad"),
    (SM, 'end - state["open_start"] >= bucket_size', 'end - state["open_start"] > bucket_size', "seal on > not >="),
    (SM, "math.lcm(dp, 128, 2**16) if busbw else math.lcm(dp, 128)", "math.lcm(dp, 128)", "busbw pad ignored"),
    (SM, "math.lcm(dp, 128, 2**16) if busbw else math.lcm(dp, 128)", "math.lcm(dp, 128, 2**16) if busbw else math.lcm(dp, 64)",
     "end pad lcm(DP, 64)"),
    (SM, '"param": local.normalize(max(0, world.start - p_start)),',
     '"param": local.normalize(max(0, p_start - world.start)),', "param view sign"),
    (SM, '        if new_bucket[pid] and state["members"]:', "        if False:", "new_bucket does not seal before"),
    (SM, "        if size_trigger or new_bucket[pid]:", "        if size_trigger:", "new_bucket does not seal after"),
    (SM, '                "shard_offset": base + local.start,', '                "shard_offset": local.start,',
     "shard offset without the bucket base"),
    (SM, "        hi = min(bucket.numel, lo + s)", "        hi = min(bucket.numel, lo + s + 1)", "slice one too long"),
    (SM, "        return sum(bk.numel // self.dp for bk in self.buffers[bi].buckets[:b])",
     "        return sum(bk.numel_unpadded // self.dp for bk in self.buffers[bi].buckets[:b])",
     "shard base from unpadded sizes"),
    (SM, '                "gbuf_world_in_bucket": Range(in_world.start - bucket.offset,',
     '                "gbuf_world_in_bucket": Range(in_world.start,', "in-bucket view not rebased"),
    (SM, '            gdt = F32 if grad_reduce_in_fp32 else p["dtype"]', '            gdt = p["dtype"]',
     "grad_reduce_in_fp32 ignored"),
    (SM, "    buf.numel_unpadded = sum(b.numel_unpadded for b in buf.buckets)",
     "    buf.numel_unpadded = sum(b.numel for b in buf.buckets)", "buffer numel_unpadded counts padding"),
]


def _copy_tree(dst):
    ignore = shutil.ignore_patterns("__pycache__", "liboracle.so*")
    for d in ("oracle", "synth"):
        shutil.copytree(os.path.join(ROOT, d), os.path.join(dst, d), ignore=ignore)
    os.makedirs(os.path.join(dst, "tests"))
    for f in ("conftest.py", "test_oracle_pins.py"):
        shutil.copy2(os.path.join(ROOT, "tests", f), os.path.join(dst, "tests", f))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(dst, "tests", "golden"))


def _run_pins(dst):
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle_pins.py", "-x", "-q",
                        "-p", "no:cacheprovider"], cwd=dst, capture_output=True, text=True, timeout=900)
    return r.returncode, r.stdout[-2000:]


def _mutant(tmp_path, i, path, old, new):
    dst = str(tmp_path / f"m{i}")
    _copy_tree(dst)
    f = os.path.join(dst, path)
    with open(f) as fh:
        src = fh.read()
    assert src.count(old) >= 1, f"mutant {i}: text not found in {path}: {old!r}"
    with open(f, "w") as fh:
        fh.write(src.replace(old, new, 1))
    rc, _ = _run_pins(dst)
    return rc


def test_every_planted_mistake_fails_a_pin(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler for the oracle")
    base = str(tmp_path / "base")
    _copy_tree(base)
    rc, out = _run_pins(base)
    assert rc == 0, "the unmutated copy must pass its pins:\n" + out
    workers = max(1, min(len(MUTANTS), os.cpu_count() or 1))
    with ThreadPoolExecutor(max_workers=workers) as pool:
        rcs = list(pool.map(lambda a: _mutant(tmp_path, *a),
                            [(i, p, o, n) for i, (p, o, n, _) in enumerate(MUTANTS)]))
    survivors = [label for (_, _, _, label), rc in zip(MUTANTS, rcs) if rc == 0]
    assert not survivors, f"mistakes no pin caught: {survivors}"
