import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the kernels)")


CHECKED_BUILD = "libdopt_checked.so"


@pytest.fixture(autouse=True)
def _bounds_record_clean(request):
    """Under the bounds-checked debug build (DOPT_LIBRARY names it), every GPU
    test must leave the kernels' bounds record empty: no tile of any launch
    fell outside its buffers."""
    yield
    if not os.environ.get("DOPT_LIBRARY", "").endswith(CHECKED_BUILD):
        return
    if request.node.get_closest_marker("gpu") is None:
        return
    import mixed_precision_adam_gb300 as D
    rec = D.dopt_debug_bounds_record()
    assert rec[0] == 0, f"kernel tiles outside their buffers: {rec[0]} checks failed, first at " \
                        f"site {rec[1]}, element {rec[2]}, extent {rec[3]}"
