import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running (still part of the default run)")


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


@pytest.fixture(scope="session")
def rlk(cuda_device):
    """The built library's binding (built in place if needed)."""
    from invariant_selected_token_gb300 import binding, build
    build.build()
    binding.lib()
    return binding


class _Qwen:
    """Qwen3-8B-shaped head (H=4096, V=151936) and the packed batch, made once per session."""

    def __init__(self, device):
        from invariant_selected_token_gb300 import workloads as WL
        self.WL = WL
        self.device = device
        self.W = WL.head_weights(device)
        self.packed = WL.packed(self.W, device)
        self._W_bits = None

    @property
    def W_bits(self):
        if self._W_bits is None:
            from invariant_selected_token_gb300 import workloads as WL
            self._W_bits = WL.bf16_tensor_bits(self.W)
        return self._W_bits


@pytest.fixture(scope="session")
def qwen(cuda_device, rlk):
    return _Qwen(cuda_device)
