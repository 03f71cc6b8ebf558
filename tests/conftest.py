import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def grpo_lib():
    """Build (if needed) and load the C-ABI library; loading needs no GPU."""
    from rl_post_token_gb300 import build as _build
    from rl_post_token_gb300 import _lib

    _build.build()
    return _lib.lib()
