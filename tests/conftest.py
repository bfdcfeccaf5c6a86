import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def load_golden(name):
    import json
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.fixture(scope="session")
def golden():
    return load_golden


@pytest.fixture
def tuning():
    """Launch-shape overrides of the library (pkv_set_tuning) for one test:
    ``tuning(decode_hpc=2)``; every knob is back to automatic afterwards."""
    import paged_kv_decode_26_gb300 as pkv
    yield pkv.set_tuning
    pkv.reset_tuning()
