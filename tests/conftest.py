import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter):
    """Parity counts per workload (rows, rows the oracle flags near a boundary, how many of those
    differ, the largest log-probability difference), as the GPU tests recorded them."""
    try:
        from _harness import REPORT
    except ImportError:
        return
    if not REPORT:
        return
    terminalreporter.write_sep("-", "parity per workload")
    for name, d in REPORT.items():
        terminalreporter.write_line(f"{name}: rows={d['rows']} flagged={d['flagged']} "
                                    f"flagged_and_different={d['flagged_and_different']} max|dlp|={d['max_dlp']:.3g}")
    path = os.environ.get("STRATA_PARITY_REPORT")
    if path:
        import json
        with open(path, "w") as f:
            json.dump(REPORT, f, indent=1)
