import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter):
    """Near-tie counts of the parity tests, by test label; also written as
    JSON to $SPEC_NEAR_TIE_REPORT when that is set."""
    try:
        from parity import NEAR_TIES
    except ImportError:
        return
    if not NEAR_TIES:
        return
    import json

    tr = terminalreporter
    tr.write_sep("-", "parity: decisions excluded as near-ties (and equally valid alternatives)")
    for label in sorted(NEAR_TIES):
        tr.write_line(f"{label}: " + ", ".join(f"{k} {v}" for k, v in sorted(NEAR_TIES[label].items())))
    path = os.environ.get("SPEC_NEAR_TIE_REPORT")
    if path:
        with open(path, "w") as f:
            json.dump(NEAR_TIES, f, indent=1, sort_keys=True)
