import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")


def load_facts():
    """Parse tests/golden/page_facts.txt into a dict of numbers."""
    facts = {}
    with open(os.path.join(ROOT, "tests", "golden", "page_facts.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = [s.strip() for s in line.split("=", 1)]
            facts[k] = float(v) if "." in v or "e" in v else int(v)
    return facts


@pytest.fixture(scope="session")
def facts():
    return load_facts()
