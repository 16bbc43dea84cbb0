import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_collection_modifyitems(config, items):
    # GPU tests are skipped (not failed) when no GPU is present, so that
    # `-m "not gpu"` and a bare run both work on a CPU-only machine.
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
    # the layer-output figures of every parity check that ran (relative Frobenius error, max-abs
    # error over rms, the bf16 rounding of the exact output alone, the bound applied)
    try:
        import _parity
    except Exception:  # pragma: no cover
        return
    if not _parity.RECORDS:
        return
    tr = terminalreporter
    tr.write_sep("-", "layer-output parity figures (max-abs and rounding in units of rms(y*))")
    tr.write_line(f"{'check':58s} {'outputs':>9s} {'rel_frob':>9s} {'max_abs':>9s} {'bf16_rnd':>9s}  bound")
    for r in _parity.RECORDS:
        tr.write_line(f"{r['label'][:58]:58s} {r['n']:9d} {r['rel_frob']:9.2e} {r['max_abs']:9.2e} "
                      f"{r['bf16_rounding']:9.2e}  {r['bound']}")
