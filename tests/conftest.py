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
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: larger CPU cases")


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
    """Print the raw errors of every GPU-vs-oracle comparison made in this session (the
    headroom under the 1e-2 / 2e-2 tolerance), and write them as JSON when PA_PARITY_REPORT
    names a file."""
    mod = sys.modules.get("parity")
    rows = getattr(mod, "REPORT", None) if mod else None
    if not rows:
        return
    tr = terminalreporter
    tr.section("parity: raw errors against the fp64 oracle (tolerance max-abs 1e-2, row max-rel 2e-2)")
    for what, n, mabs, rel in rows:
        tr.write_line(f"{mabs:10.3e} {rel:10.3e} {n:>10d}  {what}")
    worst_abs = max(r[2] for r in rows)
    worst_rel = max(r[3] for r in rows)
    tr.write_line(f"{len(rows)} comparisons; worst max-abs {worst_abs:.3e}, worst row max-rel {worst_rel:.3e}")
    out = os.environ.get("PA_PARITY_REPORT")
    if out:
        import json
        with open(out, "w") as f:
            json.dump([{"what": w, "elements": n, "max_abs": a, "max_row_rel": r} for w, n, a, r in rows], f,
                      indent=1)
