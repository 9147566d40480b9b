import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    """Run GPU tests only where a GPU is present; elsewhere skip them."""
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """One line per workload with the GPU parity statistics the tests
    gathered (code and field differences from the oracle, and how far)."""
    try:
        import _parity
    except Exception:  # pragma: no cover
        return
    if not _parity.REPORT:
        return
    import json
    tr = terminalreporter
    tr.write_sep("-", "GPU parity against the oracle, per workload")
    for name, r in sorted(_parity.REPORT.items()):
        tr.write_line(
            f"parity {name}: {r['streams']} streams, {r['codes']} codes, "
            f"{r['code_flips']} one-off codes "
            f"({r['code_flips_outside_1e3_step']} beyond 1e-3 step), "
            f"{r['field_flips']} of {r['fields']} fields differ "
            f"(max {r['field_dev_steps_max']} fp16 steps); "
            f"{r['restores']} restores, rel L2 <= {r['rel_l2_max']:.2e}, "
            f"max abs {r['max_abs']:.2e}")
    path = os.environ.get("KVTC_PARITY_REPORT")
    if path:
        with open(path, "w") as f:
            json.dump(_parity.REPORT, f, indent=1, sort_keys=True)
