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
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workloads")


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


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Prints the worst parity error of each checked quantity (tests/margins.py)."""
    import margins
    worst = margins.worst_by_quantity()
    if not worst:
        return
    tr = terminalreporter
    tr.section("parity margins (worst observed error per quantity)")
    for q in sorted(worst):
        v, b, t = worst[q]
        bound = f"bound {b:.3g}  margin x{b / v:.3g}" if (b is not None and v > 0) else (
            f"bound {b:.3g}" if b is not None else "reported")
        tr.write_line(f"{q:44s} {v:11.4g}   {bound:28s} {t}")
    if config.getoption("verbose") > 0:
        tr.section("parity margins per test")
        for t, q, v, b in margins.rows():
            tr.write_line(f"{t}  {q}: {v:.4g}" + (f" (bound {b:.3g})" if b is not None else ""))
