import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def fa_lib():
    """Build libfa.so in-tree (if stale) and return the binding module."""
    from causal_flash_attention_gb300 import build as fa_build
    fa_build.build()
    import causal_flash_attention_gb300 as fa
    fa.lib()
    return fa


@pytest.fixture(scope="module")
def fa(fa_lib):
    """The binding on a CUDA device; skips where there is none."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return fa_lib
