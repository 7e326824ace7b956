"""Shared pytest configuration.

Tests marked ``gpu`` need a CUDA device and the compiled library; everything
else runs on the CPU (oracle pins, host-side logic, library symbol checks).
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the compiled libgdn")
    config.addinivalue_line("markers", "slow: larger CPU cases")


def pytest_sessionfinish(session, exitstatus):
    """With GDN_PARITY_REPORT=<path>, write every GPU-vs-oracle comparison the
    session made (max / mean / p99 of |gpu - oracle|, violations of the
    bound) as a markdown table."""
    path = os.environ.get("GDN_PARITY_REPORT")
    if not path:
        return
    try:
        from parity_util import RECORDS
    except ImportError:
        return
    if not RECORDS:
        return
    cols = ("max_abs", "mean_abs", "p99_abs", "max_excess", "ref_max_abs", "violations", "flips")
    lines = ["| comparison | kind | bound | " + " | ".join(cols) + " |",
             "|---|---|---|" + "---|" * len(cols)]

    def fmt(v):
        if v is None:
            return ""
        if isinstance(v, (int,)) and not isinstance(v, bool):
            return str(v)
        return f"{v:.3g}"
    for r in RECORDS:
        lines.append(f"| {r['what']} | {r['kind']} | {r.get('bound') or ''} | "
                     + " | ".join(fmt(r.get(c)) for c in cols) + " |")
    with open(path, "w") as f:
        f.write("\n".join(lines) + "\n")
