import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libmtp.so")


@pytest.fixture(scope="session", autouse=True)
def _build_host_libs():
    import oracle
    import synth
    synth.build()
    oracle.build()
    yield


@pytest.fixture(scope="session")
def model27():
    """The 27B-shaped synthetic head (host arrays), built once per session."""
    import synth
    return synth.make_model(synth.QWEN27B, 2)
