import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU check")


def pytest_terminal_summary(terminalreporter):
    """The largest error / bound ratios the parity checks saw (a ratio <= 1
    passes): per-element bf16 bound and max|err|/rms against 2e-2."""
    try:
        from tests.tolerances import RECORD
    except ImportError:
        return
    if not RECORD:
        return
    tr = terminalreporter
    tr.section("parity: worst error / bound ratios")
    for kind, label in (("element", "per-element bound |err| <= 2^-8 |ref| + 1e-3 rms"),
                        ("max_rms", "max|err| / rms against 2e-2")):
        rows = sorted((r for r in RECORD if r[1] == kind), key=lambda r: -r[2])
        if not rows:
            continue
        tr.write_line(f"{label}: {len(rows)} checks, worst {rows[0][2]:.3f}")
        for what, _, ratio in rows[:5]:
            tr.write_line(f"  {ratio:.3f}  {what}")
