import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")


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


def pytest_sessionfinish(session, exitstatus):
    """Write the output-parity errors the GPU tests measured to
    $MOE_PARITY_DIR/parity_summary.json (nothing when the variable is unset)."""
    out = os.environ.get("MOE_PARITY_DIR")
    if not out:
        return
    try:
        from tests import parity
    except Exception:
        return
    if not parity.RESULTS:
        return
    import json
    os.makedirs(out, exist_ok=True)
    with open(os.path.join(out, "parity_summary.json"), "w") as f:
        json.dump([{"case": c, "max_abs_err_over_rms": a, "max_err_vs_rounded_ref_over_rms": b,
                    "elements_off_rounded_ref": n, "elements": m} for c, a, b, n, m in parity.RESULTS],
                  f, indent=1)
