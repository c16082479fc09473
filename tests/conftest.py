import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workloads")


def pytest_collection_modifyitems(config, items):
    # A gpu test on a machine without CUDA is skipped, never silently passed.
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
    """Margin of the attention parity checks to their bounds (max-abs 1e-2,
    mean-abs 1e-3): the worst cases, and every case in HB_PARITY_LOG (a JSON
    lines file) when that variable is set."""
    mod = sys.modules.get("_gpu")
    rows = getattr(mod, "MARGINS", None) if mod else None
    if not rows:
        return
    per = {}
    for test, mx, mean, xmx, xmean in rows:
        a = per.get(test, (0.0, 0.0, 0.0, 0.0))
        per[test] = (max(a[0], mx), max(a[1], mean), max(a[2], xmx), max(a[3], xmean))
    tr = terminalreporter
    tr.write_sep("-", f"attention parity margins ({len(per)} tests, {len(rows)} checks)")
    tr.write_line("of the bounds; in brackets the part beyond the exact answer's own bf16 rounding")
    worst = sorted(per.items(), key=lambda kv: -kv[1][0])[:10]
    for test, (mx, mean, xmx, xmean) in worst:
        tr.write_line(f"max-abs {mx:.2e} {100 * mx / mod.MAX_ABS:5.1f}% [{100 * xmx / mod.MAX_ABS:5.1f}%]  "
                      f"mean-abs {mean:.2e} {100 * mean / mod.MEAN_ABS:5.1f}% "
                      f"[{100 * xmean / mod.MEAN_ABS:5.1f}%]  {test}")
    path = os.environ.get("HB_PARITY_LOG")
    if path:
        import json
        with open(path, "w") as f:
            for test, (mx, mean, xmx, xmean) in sorted(per.items()):
                f.write(json.dumps({"test": test, "max_abs": mx, "mean_abs": mean,
                                    "max_abs_beyond_rounding": xmx,
                                    "mean_abs_beyond_rounding": xmean}) + "\n")
