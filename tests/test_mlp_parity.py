"""TTT-MLP: CUDA kernels vs the fp64 oracle (GPU)."""
import numpy as np
import pytest

import test_weight_sequence_ttt_b300 as ttt
from test_weight_sequence_ttt_b300.inputs import WORKLOADS, make_inputs

import torch

from _util import TOL, check_bf16_z, compare, oracle_mlp, rel_err, run_mlp, to_np

pytestmark = pytest.mark.gpu
KEYS = ("Z", "W1", "c1", "W2", "c2", "loss", "inner_loss")


def _small(d, h, b, T, B=2, H=2, io="bf16"):
    w = WORKLOADS["mlp_b4h12_d64_t8k"].with_(B=B, H=H, T=T, d=d, hidden=h, b=b, io=io, seed=91)
    return make_inputs(w)


@pytest.mark.parametrize("d,h,b,T", [(16, 64, 4, 32), (64, 256, 16, 48), (32, 128, 1, 12)])
def test_mlp_f32(d, h, b, T):
    inp = _small(d, h, b, T, io="f32")
    got = run_mlp(inp)
    assert int(got["status"].item()) == 0
    compare(got, oracle_mlp(inp), KEYS, TOL["f32"])


@pytest.mark.parametrize("d,h,b,T", [(64, 256, 16, 64), (64, 256, 4, 40)])
def test_mlp_bf16(d, h, b, T):
    inp = _small(d, h, b, T)
    got = run_mlp(inp)
    assert int(got["status"].item()) == 0
    compare(got, oracle_mlp(inp), KEYS, TOL["bf16"])


def test_mlp_bf16_z_output():
    inp = _small(64, 256, 16, 32)
    got = run_mlp(inp, z_dtype=torch.bfloat16)
    check_bf16_z(got["Z"], oracle_mlp(inp)["Z"], TOL["bf16"])


def test_mlp_full_size_sampled_chains():
    w = WORKLOADS["mlp_b4h12_d64_t8k"]
    inp = make_inputs(w)
    got = run_mlp(inp)
    assert int(got["status"].item()) == 0
    sel = [0, w.chains - 1]
    ref = oracle_mlp(make_inputs(w, chains=sel))
    idx = (np.array([c // w.H for c in sel]), np.array([c % w.H for c in sel]))
    errs = {k: rel_err(to_np(got[k])[idx], ref[k].reshape(to_np(got[k])[idx].shape)) for k in KEYS}
    print(errs)
    assert errs["Z"] <= TOL["bf16"], errs
