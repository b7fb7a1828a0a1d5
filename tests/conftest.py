import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libkvm.so")


@pytest.fixture(scope="session", autouse=True)
def _oracle_built():
    import oracle
    oracle.build()
    yield


def pytest_sessionfinish(session, exitstatus):
    """Write the near-tie counts the GPU parity tests collected (if any ran)."""
    import json
    import kvm_testlib
    if not kvm_testlib.REPORT:
        return
    out = os.path.join(HERE, "reports")
    os.makedirs(out, exist_ok=True)
    with open(os.path.join(out, "near_ties.json"), "w") as f:
        json.dump({"near_tie_threshold": kvm_testlib.NEAR_TIE,
                   "workloads": kvm_testlib.REPORT}, f, indent=1, sort_keys=True)
