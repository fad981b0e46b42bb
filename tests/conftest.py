import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def page_facts():
    with open(os.path.join(ROOT, "tests", "golden", "page_facts.json")) as f:
        return {k: v["value"] for k, v in json.load(f).items() if not k.startswith("_")}
