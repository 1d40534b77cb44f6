import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.dirname(os.path.abspath(__file__))
for _p in (ROOT, TESTS):
    if _p not in sys.path:
        sys.path.insert(0, _p)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (a GB300, sm_103)")


def load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.fixture
def golden():
    return load_golden


def pytest_terminal_summary(terminalreporter):
    """Prints the literal errors of every GPU-vs-oracle comparison this session made."""
    parity = sys.modules.get("parity")
    records = getattr(parity, "RECORDS", None) if parity else None
    if not records:
        return
    terminalreporter.section("parity against the float64 oracle")
    for label, rec in records:
        terminalreporter.write_line(parity.format_record(label, rec))
