"""Shared pytest set-up: the `gpu` marker and import paths.

CLK_TEST_LIBRARY (environment) points the binding at another build of the
library, e.g. the reduced-fingerprint build that
test_gpu_fingerprint_collisions.py makes and runs the parity tests against."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

_ALT_LIB = os.environ.get("CLK_TEST_LIBRARY")
if _ALT_LIB:
    import context_lookup_speculative_gb300 as _clk

    if not os.path.exists(_ALT_LIB):
        raise RuntimeError(f"CLK_TEST_LIBRARY={_ALT_LIB} does not exist")
    _clk.LIB_PATH = _ALT_LIB


def pytest_report_header(config):
    return f"clk library under test: {_ALT_LIB}" if _ALT_LIB else None


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")
