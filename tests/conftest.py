import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:                                   # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device in this process")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Print the routing and sampled-parity records the GPU tests kept, so that
    near ties, flips and float errors are visible in a quiet (-q) run."""
    mod = sys.modules.get("parity")
    recs = getattr(mod, "REPORT", None) if mod else None
    if not recs:
        return
    terminalreporter.section("parity records")
    for r in recs:
        terminalreporter.write_line(" ".join(f"{k}={v:.3g}" if isinstance(v, float) else f"{k}={v}"
                                             for k, v in sorted(r.items())))
