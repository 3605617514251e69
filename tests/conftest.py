import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the CUDA library")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes of oracle time)")


@pytest.fixture(scope="session", autouse=True)
def _host_libs():
    """Builds the generator and the oracle (gcc, seconds) once per session."""
    import oracle
    import synth
    synth.build()
    oracle.build()
