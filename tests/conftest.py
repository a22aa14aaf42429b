import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running (full-size workloads)")


def pytest_collection_modifyitems(config, items):
    try:
        import torch

        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_runtest_logreport(report):
    """With INK_TEST_LOG set, append every test's outcome and duration to that file as it finishes."""
    path = os.environ.get("INK_TEST_LOG")
    if not path or report.when != "call" and not (report.when == "setup" and report.outcome != "passed"):
        return
    with open(path, "a") as f:
        f.write(f"{report.outcome:8s} {report.duration:8.2f}s {report.nodeid}\n")
        if report.outcome == "failed":
            f.write(str(report.longrepr)[-3000:] + "\n")
