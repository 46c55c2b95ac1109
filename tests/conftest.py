import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")


def pytest_collection_modifyitems(config, items):
    # GPU tests are skipped (not failed) when no CUDA device is visible, so a
    # plain `pytest tests/` on a CPU-only machine stays green.
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
    """Selected-page parity of the GPU tests: how many (sequence, KV head)
    units were compared with the oracle, every page decided differently (each
    inside its ε_sel or bf16 rounding band, else its test failed), and the
    smallest float64 decision margin met."""
    h = sys.modules.get("harness")
    if h is None or not h.PARITY["checks"]:
        return
    p = h.PARITY
    tr = terminalreporter
    tr.write_line(f"selected-page parity: {p['checks']} decodes, {p['units']} (sequence, KV head) units, "
                  f"{p['pages']} page decisions, {len(p['flips'])} flips")
    if p["min_margin_at"] is not None:
        tr.write_line(f"smallest |decision margin|: {p['min_margin']:.3e} at {p['min_margin_at']}")
    for f in p["flips"]:
        tr.write_line("  flip " + f)
