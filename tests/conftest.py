import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size parity case (minutes of oracle time)")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


@pytest.fixture(autouse=True)
def _device_error_word_clean(request):
    """After every GPU test, no kernel may have reported a failed bounded wait
    or a failed internal count check."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import activation_sparse_gb300 as si
    code = si.si_device_error(clear=True)
    assert code == 0, "device error word = %#x" % code
