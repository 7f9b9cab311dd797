"""The GPU tests again, through the bounds-checked debug build of the library
(lib/libdopt_checked.so, compiled with DOPT_BOUNDS_CHECK=1): every kernel of
that build checks each tile's element ranges against the extents of the
buffers it reads and writes and records any that fall outside (skipping the
tile), and the conftest fixture fails a test whose launches left such a
record.  Together with the parity comparisons this stands in for a memory
checker: every access of every tested launch, full sizes included, stayed
inside its buffer."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CHECKED = os.path.join(ROOT, "mixed_precision_adam_gb300", "lib", "libdopt_checked.so")
FILES = ["test_parity_gpu.py", "test_random_gpu.py", "test_fullsize_gpu.py", "test_bucket_staged_gpu.py",
         "test_grad_check_gpu.py", "test_graph_gpu.py", "test_from_host_gpu.py", "test_state_model_gpu.py",
         "test_memory_gpu.py", "test_multirank_device_gpu.py", "test_zz_no_alloc.py"]


def test_gpu_suite_under_the_bounds_checked_build():
    if not os.path.exists(CHECKED):
        sys.path.insert(0, os.path.join(ROOT, "mixed_precision_adam_gb300"))
        import build
        build.build_checked()
    env = dict(os.environ, DOPT_LIBRARY=CHECKED)
    out = subprocess.run([sys.executable, "-m", "pytest", *[os.path.join(ROOT, "tests", f) for f in FILES],
                          "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider"],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert out.returncode == 0, out.stdout[-4000:] + out.stderr[-2000:]
    assert " passed" in out.stdout
