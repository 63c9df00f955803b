import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Seed redraws of the GPU parity runs: rounds whose oracle decision gaps fell below 1e-5
    relative were redrawn (new generator salt) before being compared; the counts are reported."""
    harness = sys.modules.get("harness")
    log = getattr(harness, "REDRAW_LOG", None)
    if not log:
        return
    tr = terminalreporter
    tr.section("seed redraws (oracle decision gap < 1e-5 relative)")
    tot_r = tot_q = tot_h = 0
    for label, rounds, redrawn, hit in log:
        tr.write_line(f"{label}: {rounds} rounds compared, {hit} redrawn, {redrawn} request redraws")
        tot_r, tot_q, tot_h = tot_r + rounds, tot_q + redrawn, tot_h + hit
    tr.write_line(f"total: {tot_r} rounds compared, {tot_h} redrawn, {tot_q} request redraws")
    cache = getattr(config, "cache", None)
    if cache is not None:
        cache.set("dt/seed_redraws", {"runs": [list(x) for x in log],
                                      "total": {"rounds": tot_r, "rounds_redrawn": tot_h,
                                                "request_redraws": tot_q}})
