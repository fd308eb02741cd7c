import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_collection_modifyitems(config, items):
    # GPU tests are skipped, not failed, where no GPU is present.
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
    """Every bf16 output compared with the oracle in this run: the literal
    max|err|/rms(ref) (bar 2e-2), mean relative error (5e-3), the worst
    element's error over its bar and how many elements are beyond 2e-2 rms
    (only possible where bf16 cannot resolve the bar)."""
    from tests.util import PARITY_LOG
    if not PARITY_LOG:
        return
    tr = terminalreporter
    tr.write_line(f"parity vs oracle ({len(PARITY_LOG)} comparisons): max|err|/rms  mean_rel  worst/bar"
                  "  n(err > 2e-2 rms)")
    worst = max(PARITY_LOG, key=lambda r: r[1])
    for what, mx, mr, wb, nl in PARITY_LOG:
        tr.write_line(f"  {what[:48]:48s} {mx:.5f}  {mr:.2e}  {wb:.3f}  {nl}")
    tr.write_line(f"parity worst max|err|/rms: {worst[1]:.5f} ({worst[0]})")
