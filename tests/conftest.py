import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")


def pytest_collection_modifyitems(config, items):
    # GPU tests are skipped, not failed, when no device is visible.
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """The literal max-abs figures: largest max |y - y_ref| / rms(y_ref) over every
    BF16-output comparison (bounded per element with a half-ulp allowance) and over
    every FP32-output comparison (bounded literally by 1e-2)."""
    try:
        from helpers import LITERAL_LOG
    except ImportError:
        return
    if not LITERAL_LOG:
        return
    tr = terminalreporter
    tr.section("output error vs the FP64 oracle (literal max-abs)")
    for fp32 in (False, True):
        rows = [r for r in LITERAL_LOG if r[3] == fp32]
        if not rows:
            continue
        worst_lit = max(rows, key=lambda r: r[2])
        worst_rel = max(rows, key=lambda r: r[1])
        kind = "FP32 outputs" if fp32 else "BF16 outputs"
        tr.write_line(f"{kind}: {len(rows)} comparisons; max |err|/rms = {worst_lit[2]:.3e} ({worst_lit[0]}); "
                      f"max relL2 = {worst_rel[1]:.3e} ({worst_rel[0]})")
