import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")
    # (re)build libkvattn.so if any source is newer than it; a no-op otherwise.
    # build.py is loaded by path: importing the package would load the library.
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_kvattn_build", os.path.join(ROOT, "continuous_batching_kv_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()


def golden(name):
    import json
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.fixture
def gold():
    return golden


def pytest_terminal_summary(terminalreporter):
    """Worst attention error per GPU test against the tolerance (max-abs 2e-3,
    rel-L2 1e-2), so that the margin is on record in the run's output."""
    try:
        from tests.gpu_util import MARGINS
    except Exception:
        return
    if not MARGINS:
        return
    tr = terminalreporter
    tr.write_line("worst attention error per test (max-abs / rel-L2 / outputs compared):")
    for name, (a, r, n) in sorted(MARGINS.items()):
        tr.write_line("  %-58s %.2e  %.2e  %d" % (name[:58], a, r, n))
