import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def read_golden(name):
    """Non-comment, non-empty lines of a golden fixture, split on whitespace."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


@pytest.fixture
def golden():
    return read_golden


def pytest_terminal_summary(terminalreporter):
    """Worst attention errors seen against the oracle (the margins under the
    tolerances) and the tests that produced them, when any comparison ran."""
    parity = sys.modules.get("tests.parity")
    errs = getattr(parity, "ERRORS", None)
    if errs:
        rel = max(e[0] for e in errs)
        mx = max(e[1] for e in errs)
        terminalreporter.write_line(
            f"attention parity: {len(errs)} comparisons, worst rel-L2 {rel:.3e} (limit {parity.REL_L2:g}), "
            f"worst max-abs {mx:.3e} (limit {parity.MAX_ABS:g})")
        worst = {}
        for e in errs:
            name = e[2].split("[")[0]
            if name not in worst or e[0] > worst[name][0]:
                worst[name] = e
        for e in sorted(worst.values(), key=lambda e: -e[0]):
            terminalreporter.write_line(f"  rel-L2 {e[0]:.3e}  max-abs {e[1]:.3e}  {e[2]}")
