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
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """The accuracy margins of the full-size parity tests: per workload and
    kernel, the worst max|err| / max|V| over every output compared, next to
    its gate."""
    helpers = sys.modules.get("tests.helpers")
    margins = getattr(helpers, "MARGINS", None) if helpers else None
    if not margins:
        return
    terminalreporter.write_line("accuracy margins (worst max|err| / max|V|, gate):")
    for label in sorted(margins):
        r, tol = margins[label]
        terminalreporter.write_line(f"  {label}: {r:.3e} (gate {tol:.0e}, {r / tol:.3f} of it)")
