import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: longer CPU statistics")


def read_facts(name):
    """Parse a tests/golden/*.txt fact file into {key: [list of value lists]}."""
    facts = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            facts.setdefault(key, []).append(vals)
    return facts


@pytest.fixture(scope="session")
def mask_facts():
    return read_facts("mask_page_facts.txt")


@pytest.fixture(scope="session")
def verifier_facts():
    return read_facts("verifier_page_facts.txt")
