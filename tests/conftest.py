import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long CPU-only oracle runs")
    config.addinivalue_line("markers", "fullsize: GPU parity over a whole benchmark launch "
                            "(minutes of oracle time; still part of -m gpu)")


def pytest_collection_modifyitems(config, items):
    import torch
    if torch.cuda.is_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """Print the skip-bit flips of every GPU/oracle bitmap comparison: blocks
    whose bit differs, out of the blocks whose oracle statistic lies in the
    margin band around ln(lambda), out of the traversed blocks."""
    try:
        from tests.parity import FLIP_LOG
    except Exception:
        return
    if not FLIP_LOG:
        return
    tr = terminalreporter
    tr.section("skip-bit flips inside the margin band")
    flips = sum(f for _, f, _, _ in FLIP_LOG)
    near = sum(n for _, _, n, _ in FLIP_LOG)
    trav = sum(t for _, _, _, t in FLIP_LOG)
    tr.write_line(f"{len(FLIP_LOG)} comparisons: {flips} flips, {near} blocks in the band, "
                  f"{trav} traversed blocks")
    for label, f, n, t in FLIP_LOG:
        if f or n:
            tr.write_line(f"  {label}: {f} flips / {n} in band / {t} traversed")
