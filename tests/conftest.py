import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_sessionfinish(session, exitstatus):
    """Write the parity records (excused decisions, K/V error ratios) the GPU
    tests collected: to $MTP_PARITY_REPORT, else gpurun_out/parity_report.json
    under the repository root.  Nothing is written when no GPU test ran."""
    from parity_helpers import write_report
    path = os.environ.get("MTP_PARITY_REPORT") or os.path.join(ROOT, "gpurun_out", "parity_report.json")
    write_report(path)
