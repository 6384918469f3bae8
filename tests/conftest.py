import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built extension")


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


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """The near-boundary counts of the matching rules, per parity case: requests compared, requests
    whose draw lay within 1e-6 of a decision boundary (flagged), and requests whose GPU output
    differed from the oracle's (allowed only when flagged, and fewer than 0.01% of requests)."""
    parity = sys.modules.get("parity")
    counts = getattr(parity, "COUNTS", None)
    if not counts:
        return
    tr = terminalreporter
    tr.write_sep("-", "near-boundary counts (requests / flagged / mismatched)")
    tot = [0, 0, 0]
    for label in sorted(counts):
        n, f, m = counts[label]
        tot = [tot[0] + n, tot[1] + f, tot[2] + m]
        tr.write_line(f"{label:<40s} {n:>8d} {f:>6d} {m:>6d}")
    tr.write_line(f"{'all':<40s} {tot[0]:>8d} {tot[1]:>6d} {tot[2]:>6d}  "
                  f"(mismatched {100.0 * tot[2] / max(tot[0], 1):.4f}% of requests)")
