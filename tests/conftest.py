import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size parity case")


def _cuda_ok():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if _cuda_ok():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


@pytest.fixture(params=[0, 2], ids=["one_cta", "cluster"])
def linear_form(request):
    """Runs a test with each form of the d = 64, mb = 16 TTT-Linear kernel: one
    CTA per chain (0) and the two-CTA cluster per chain (2); other shapes are
    unaffected. The default (0) comes back afterwards."""
    import test_weight_sequence_ttt_b300 as ttt
    ttt.linear_cluster_mode(request.param)
    yield request.param
    ttt.linear_cluster_mode(0)


@pytest.fixture(params=[0, 2], ids=["one_cta", "cluster"])
def mlp_form(request):
    """Runs a test with each form of the tensor-core TTT-MLP kernel: one CTA per
    chain (0) and the two-CTA cluster with the hidden units split (2). The
    default (1: the cluster when the chains fit half the SMs) comes back
    afterwards."""
    import test_weight_sequence_ttt_b300 as ttt
    ttt.mlp_cluster_mode(request.param)
    yield request.param
    ttt.mlp_cluster_mode(1)
