import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libkvsel.so")
    config.addinivalue_line("markers", "slow: long-running case (full-size oracle comparison)")
    # libkvsel.so and the oracle are built in-tree (only when stale) before collection
    import __graft_entry__
    __graft_entry__.load_builder().build()
    import oracle
    oracle.build()


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture
def golden():
    import json

    def load(name):
        with open(os.path.join(GOLDEN, name)) as f:
            return json.load(f)

    return load
