import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a); runs the CUDA path through the C-ABI")


def has_gpu() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def gpu_lib():
    """The C-ABI library, loaded; skips the test only when no GPU is present."""
    if not has_gpu():
        pytest.skip("no CUDA device")
    import dense_attention_forward_fwd_gb300 as attn
    attn.load_library()
    return attn
