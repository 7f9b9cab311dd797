"""The ctypes binding's structs must match include/dopt.h byte for byte: a
small C program compiled with the system compiler prints every struct's size
and field offsets, and the test compares them with the binding's."""

import ctypes
import os
import shutil
import subprocess

import pytest

dopt = pytest.importorskip("mixed_precision_adam_gb300")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
STRUCTS = ["dopt_range", "dopt_param_desc", "dopt_buffer_info", "dopt_bucket_info",
           "dopt_param_shard", "dopt_adamw_hparams", "dopt_step_args", "dopt_step_stats",
           "dopt_loss_scaler"]


def test_binding_structs_match_header(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "dopt.h"', "int main(void) {"]
    for name in STRUCTS:
        lines.append(f'  printf("{name} size %zu\\n", sizeof({name}));')
        for field, _ in getattr(dopt, name)._fields_:
            lines.append(f'  printf("{name} {field} %zu\\n", offsetof({name}, {field}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    for line in filter(None, out):
        name, what, value = line.split()
        cls = getattr(dopt, name)
        got = ctypes.sizeof(cls) if what == "size" else getattr(cls, what).offset
        assert got == int(value), (name, what, got, value)
