import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_sessionfinish(session, exitstatus):
    """Write every parity comparison of the session to $NF_PARITY_LOG (JSON)
    and a per-test summary table beside it ($NF_PARITY_LOG with .md)."""
    path = os.environ.get("NF_PARITY_LOG")
    if not path:
        return
    import json
    try:
        from tests.helpers import RECORD
    except Exception:  # pragma: no cover
        return
    with open(path, "w") as f:
        json.dump(RECORD, f, indent=0)
    worst = {}
    for r in RECORD:
        key = (r["test"].split("::")[-1], r["name"].split(",")[0], r["oracle"])
        w = worst.setdefault(key, dict(r, count=0))
        w["count"] += 1
        for k in ("max_abs", "rel_l2"):
            w[k] = max(w[k], r[k])
    lines = ["| test | output | oracle | checks | elements | max-abs | rel-L2 | rms(ref) |",
             "|---|---|---|---|---|---|---|---|"]
    for (test, name, oracle), w in worst.items():
        lines.append(f"| {test} | {name} | {oracle} | {w['count']} | {w['n']} | {w['max_abs']:.4g} | "
                     f"{w['rel_l2']:.3g} | {w['rms_ref']:.3g} |")
    with open(os.path.splitext(path)[0] + ".md", "w") as f:
        f.write("\n".join(lines) + "\n")
