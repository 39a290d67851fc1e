import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libkda")


@pytest.fixture(scope="session")
def kda():
    """The CUDA binding; built once per session (on the GPU machine the build happens here too)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_26_gb300 import build as _build
    _build.build()
    from gated_delta_rule_26_gb300 import kda as _kda
    return _kda
