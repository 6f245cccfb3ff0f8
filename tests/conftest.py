import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: takes more than a few seconds")


def pytest_report_header(config):
    """The library version and source hash this run tests (if it is built)."""
    try:
        from blackwell_tensor_core_gb300 import build
        v = build.built_version()
        return "bwgemm: %s (sources on disk: %s)" % (v or "not built", build.source_hash())
    except Exception as e:  # noqa: BLE001 - a header line must not fail the run
        return "bwgemm: version unavailable (%s)" % e
