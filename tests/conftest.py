import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")


@pytest.fixture
def gemm_switch():
    """set(cta2, wide) sets libkd's GEMM tile switches (kd_test_set_gemm_tiles;
    -1 or None = the default) for one test; the defaults come back after it."""
    from top_kl_loss_tcgen05_b300 import _native

    def set_(cta2, wide=None):
        _native.set_gemm_tiles(-1 if cta2 is None else int(cta2), -1 if wide is None else int(wide))

    yield set_
    _native.set_gemm_tiles(-1, -1)


@pytest.fixture
def topk_exact():
    """set(on) sends every top-K row through the exact radix selection
    (kd_test_set_topk_force_exact) for one test; the default comes back after it."""
    from top_kl_loss_tcgen05_b300 import _native

    yield _native.set_topk_force_exact
    _native.set_topk_force_exact(False)


@pytest.fixture(scope="session")
def cuda_dev():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")
