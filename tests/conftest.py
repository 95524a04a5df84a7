import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    # GPU tests are skipped, not failed, when no GPU is visible, so that
    # `-m "not gpu"` and a plain run on a CPU host both stay green.
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device visible")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Near-tie report of the GPU parity checks: per test, the units compared,
    the size of the exemption band E (positions whose oracle pooled score is
    within 1e-5 relative of the (C-W)-th best) and how many positions in E
    were kept by only one side.  Written as JSON too when
    SNAPKV_PARITY_REPORT names a file."""
    mod = sys.modules.get("tests.parity")
    rows = getattr(mod, "NEAR_TIES", None) if mod else None
    if not rows:
        return
    tr = terminalreporter
    tr.section("near-tie exemptions (GPU vs oracle)")
    tr.write_line(f"{'units':>6} {'|E|':>6} {'kept by one side':>16}  test")
    for r in rows:
        tr.write_line(f"{r['units']:>6} {r['band']:>6} {r['decided_in_band']:>16}  {r['test']}")
    tot = {k: sum(r[k] for r in rows) for k in ("units", "band", "decided_in_band")}
    tr.write_line(f"{tot['units']:>6} {tot['band']:>6} {tot['decided_in_band']:>16}  (total, "
                  f"{len(rows)} checks)")
    path = os.environ.get("SNAPKV_PARITY_REPORT")
    if path:
        import json
        with open(path, "w") as f:
            json.dump({"checks": rows, "total": tot}, f, indent=1)
