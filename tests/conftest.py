import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU case")


def pytest_terminal_summary(terminalreporter):
    """The recorded parity margins of every float comparison that ran, worst case per
    label: max|err|/RMS against the 2e-2 bound (before the allowances), relative L1
    against 5e-3, the largest MXFP8-h ambiguity slack (fraction of RMS), the share of
    elements that needed it, and the share whose error exceeded 2e-2 * RMS at all (the
    bf16 half-ulp of large outputs and the ambiguity slack explain those)."""
    from tests._util import MARGINS
    if not MARGINS:
        return
    groups = {}
    for m in MARGINS:
        groups.setdefault(m["what"], []).append(m)
    tr = terminalreporter
    tr.write_sep("-", "parity margins (max|err|/RMS <= 2e-2, rel L1 <= 5e-3), worst per label")
    for what, ms in groups.items():
        tr.write_line(f"{what:<52} x{len(ms):<4} max|err|/rms {max(m['max_err_rms'] for m in ms):.3e}  "
                      f"relL1 {max(m['rel_l1'] for m in ms):.3e}  "
                      f"slack/rms {max(m['max_slack_rms'] for m in ms):.2e} "
                      f"(needed by {max(m['slack_frac'] for m in ms):.1e})  "
                      f"over 2e-2*rms {max(m['bf16_frac'] for m in ms):.1e}")
