import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


import pytest  # noqa: E402


@pytest.fixture
def plan_overrides():
    """Set the library's plan overrides (the rnn_debug_set_plan_overrides test
    hook) for one test; they are cleared afterwards."""
    import bwd_persistent_cta_gb300 as R

    def set_(**kw):
        rc = R.rnn_debug_set_plan_overrides(**kw)
        assert rc == R.RNN_OK, R.rnn_status_string(rc)

    yield set_
    R.rnn_debug_set_plan_overrides()
