"""Shared test set-up: repo root on sys.path, the gpu marker, device helpers."""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library binding; only gpu tests ask for it."""
    import torch

    if not torch.cuda.is_available():
        pytest.fail("gpu test collected without a CUDA device")
    import quantized_expert_ffn_router_gb300 as ft

    ft.load()
    return ft
