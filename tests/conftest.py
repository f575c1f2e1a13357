import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libssscan.so")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes of oracle time)")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Observed parity errors of the session: the largest per (test file, tensor), both metrics; written in
    full as JSON to $PARITY_REPORT when that is set."""
    from tests._util import RECORD
    if not RECORD:
        return
    worst = {}
    for node, name, e, el in RECORD:
        key = (node.split("::")[0], name)
        a, b = worst.get(key, (0.0, 0.0))
        worst[key] = (max(a, e), max(b, el))
    tr = terminalreporter
    tr.write_line(f"parity: {len(RECORD)} comparisons; largest observed error per (file, tensor): "
                  "inf-norm relative | elementwise over |r| >= 1e-2 max|r|")
    for (f, name), (e, el) in sorted(worst.items()):
        tr.write_line(f"  {f:38s} {name:14s} {e:.2e} | {el:.2e}")
    path = os.environ.get("PARITY_REPORT")
    if path:
        import json
        with open(path, "w") as fh:
            json.dump([{"test": n, "tensor": t, "inf_rel": e, "elem_rel": el} for n, t, e, el in RECORD], fh, indent=0)
