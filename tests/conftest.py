import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    # temporary files of the tests (tmp_path) stay inside the checkout, in a git-ignored folder
    # that pytest clears at the start of each session
    if getattr(config.option, "basetemp", None) is None:
        os.makedirs(os.path.join(ROOT, "_build"), exist_ok=True)
        config.option.basetemp = os.path.join(ROOT, "_build", "pytest-tmp")
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: generates full-size workloads on the host")


_WORKLOAD_CACHE = {}


@pytest.fixture(scope="session")
def workload():
    """Session cache of the five seeded workloads (generation of c4 takes seconds)."""
    import workloads

    def get(name):
        if name not in _WORKLOAD_CACHE:
            _WORKLOAD_CACHE[name] = workloads.make(name)
        return _WORKLOAD_CACHE[name]

    return get
