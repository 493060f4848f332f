import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")


def gpu_available():
    try:
        import torch

        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if gpu_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """One JSON line per workload whose routing the GPU parity tests checked:
    its token count, how many tokens were near-ties (oracle margin <= 1e-5,
    validity-checked instead of compared id by id) and how many outputs were
    compared with the oracle."""
    helpers = sys.modules.get("parity_helpers")
    records = getattr(helpers, "NEAR_TIES", None) if helpers is not None else None
    if not records:
        return
    terminalreporter.section("routing near-ties per workload")
    for rec in records:
        terminalreporter.write_line("near_ties " + json.dumps(rec))
