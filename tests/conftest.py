import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workloads (seconds to minutes)")


def pytest_collection_modifyitems(config, items):
    # GPU tests cannot run without a device; skip them loudly rather than let
    # them fail on a CPU-only host when selected explicitly.
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device on this host")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """How often the GPU parity checks needed their floors: dx elements
    within the cancellation floor but not within 1 ulp (or fp32's relative
    bound), and parameter-gradient columns within the summation floor but
    not the relative bound."""
    try:
        import helpers
    except Exception:
        return
    tr = terminalreporter
    if helpers.FLOOR_USES:
        tot = sum(e for _, e, _ in helpers.FLOOR_USES)
        used = sum(n for _, _, n in helpers.FLOOR_USES)
        worst = max(helpers.FLOOR_USES, key=lambda r: r[2] / max(r[1], 1))
        tr.write_line(f"dx cancellation floor: {used} of {tot} elements over {len(helpers.FLOOR_USES)} checks "
                      f"({used / max(tot, 1) * 1e6:.2f} per million); highest share {worst[2]} of {worst[1]} "
                      f"in {worst[0]}")
    if helpers.DW_FLOOR_USES:
        cols = sum(c for _, c, _, _ in helpers.DW_FLOOR_USES)
        used = sum(n for _, _, n, _ in helpers.DW_FLOOR_USES)
        worst = max(helpers.DW_FLOOR_USES, key=lambda r: r[3])
        tr.write_line(f"parameter-gradient summation floor: {used} of {cols} columns over "
                      f"{len(helpers.DW_FLOOR_USES)} checks; worst error {worst[3]:.3f} of the relative bound "
                      f"in {worst[0]}")
