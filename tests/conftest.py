import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_terminal_summary(terminalreporter):
    """Totals of the GPU parity checks: codes compared, in-band ties, output
    elements compared, end-to-end checks left out because of ties."""
    mod = sys.modules.get("vqcase")
    if mod is None or not any(mod.CHECKS.values()):
        return
    c = mod.CHECKS
    terminalreporter.write_line(
        f"parity: {c['codes']} codes compared, {c['code_ties']} in-band ties; {c['outputs']} output "
        f"elements compared; {c['e2e_skipped']} end-to-end checks left out for ties")
    for line in mod.PARITY_NOTES:
        terminalreporter.write_line("  " + line)
