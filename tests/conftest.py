import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_terminal_summary(terminalreporter):
    """Report the near-tie bucket mismatches every parity case counted: each one lies
    inside the band where the oracle's top-1/top-2 projection margin is below
    1e-5 * |x| * |R|, the only place a mismatch is allowed."""
    mod = sys.modules.get("tests.parity")
    rec = getattr(mod, "NEAR_TIES", None)
    if not rec:
        return
    tr = terminalreporter
    tr.write_sep("-", "near-tie bucket mismatches (all inside the 1e-5*|x|*|R| band)")
    for case in sorted(rec):
        bad, tot = rec[case]
        tr.write_line(f"{case}: {bad} of {tot} buckets ({bad / max(tot, 1):.2e})")
