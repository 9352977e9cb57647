import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


@pytest.fixture(scope="session")
def torch_cuda():
    """torch with CUDA initialised and the library built and loaded."""
    import torch

    import sparse_attention_decode_msa_gb300 as msa
    from sparse_attention_decode_msa_gb300 import build

    build.build()
    msa.load()
    torch.cuda.init()
    return torch


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    # Keep GPU tests off machines without a GPU even if the marker filter is not given.
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)
