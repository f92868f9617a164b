import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built extension")
    config.addinivalue_line("markers", "slow: full-size parity cases")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Raw attention errors per test against the stated flat bars (max-abs
    2e-2, rel-L2 1e-2), and the largest share of the derived per-element
    limit that any element used. With CSA2_PARITY_REPORT set, the same rows
    are written to that path as JSON."""
    gc = sys.modules.get("gpu_common")
    log = getattr(gc, "PARITY_LOG", None) if gc is not None else None
    if not log:
        return
    per = {}
    for test, what, max_abs, rel, used, n_over, n in log:
        r = per.setdefault(test, dict(test=test, checks=0, max_abs=0.0, rel_l2=0.0, limit_used=0.0,
                                      over_flat=0, elements=0))
        r["checks"] += 1
        r["max_abs"] = max(r["max_abs"], max_abs)
        r["rel_l2"] = max(r["rel_l2"], rel)
        r["limit_used"] = max(r["limit_used"], used)
        r["over_flat"] += n_over
        r["elements"] += n
    tr = terminalreporter
    tr.section("attention parity: raw errors against max-abs 2e-2 / rel-L2 1e-2")
    tr.write_line(f"{'test':<70} {'checks':>6} {'max-abs':>10} {'rel-L2':>10} {'>2e-2':>8} {'limit used':>10}")
    for r in per.values():
        tr.write_line(f"{r['test'][-70:]:<70} {r['checks']:>6} {r['max_abs']:>10.3e} {r['rel_l2']:>10.3e} "
                      f"{r['over_flat']:>8} {r['limit_used']:>10.3f}")
    path = os.environ.get("CSA2_PARITY_REPORT")
    if path:
        with open(path, "w") as f:
            json.dump(list(per.values()), f, indent=1)
