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
def test_mlp_bf16(d, h, b, T, mlp_form):
    inp = _small(d, h, b, T)
    got = run_mlp(inp)
    assert int(got["status"].item()) == 0
    compare(got, oracle_mlp(inp), KEYS, TOL["bf16"])


def test_mlp_bf16_z_output(mlp_form):
    inp = _small(64, 256, 16, 32)
    got = run_mlp(inp, z_dtype=torch.bfloat16)
    check_bf16_z(got["Z"], oracle_mlp(inp)["Z"], TOL["bf16"])


def test_mlp_full_size_sampled_chains(mlp_form):
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
    for k in KEYS:
        assert errs[k] <= 5 * TOL["bf16"], errs


def test_mlp_full_size_bf16_z_matches_fp32_z(mlp_form):
    """bf16 Z (the kernels instantiated for the standard flags) against fp32 Z (the
    general ones) at the benchmark size: the same state and losses bit for bit, and
    Z the round-to-nearest-even bf16 of the fp32 Z."""
    w = WORKLOADS["mlp_b4h12_d64_t8k"]
    inp = make_inputs(w)
    a = run_mlp(inp, z_dtype=torch.bfloat16)
    b = run_mlp(inp, z_dtype=torch.float32)
    assert int(a["status"].item()) == 0 and int(b["status"].item()) == 0
    for k in ("W1", "c1", "W2", "c2", "loss", "inner_loss"):
        assert torch.equal(a[k], b[k]), k
    assert torch.equal(a["Z"], b["Z"].to(torch.bfloat16))


# ---------------------------------------------------------------- tensor-core MLP kernel (d=64, h=256, b=16)

def _tc(T=64, B=2, H=2, seed=91):
    w = WORKLOADS["mlp_b4h12_d64_t8k"].with_(B=B, H=H, T=T, seed=seed)
    return make_inputs(w)


def test_mlp_tc_kernel_kind():
    assert ttt.mlp_kernel_kind(ttt.BF16, 64, 256, 16) == 2
    assert ttt.mlp_kernel_kind(ttt.BF16, 64, 256, 4) == 1
    assert ttt.mlp_kernel_kind(ttt.F32, 64, 256, 16) == 1


@pytest.mark.parametrize("T", [16, 32, 160])
def test_mlp_tc_lengths(T, mlp_form):
    inp = _tc(T=T, B=1, H=3)
    got = run_mlp(inp)
    assert int(got["status"].item()) == 0
    compare(got, oracle_mlp(inp), KEYS, TOL["bf16"])


def test_mlp_tc_per_sequence_weights_and_ln_params(mlp_form):
    inp = _tc(T=48, B=3, H=2)
    g = torch.Generator().manual_seed(11)
    inp["W1"] = torch.randn(3, 2, 256, 64, generator=g) * 0.05
    inp["W2"] = torch.randn(3, 2, 64, 256, generator=g) * 0.05
    inp["c1"] = torch.randn(3, 2, 256, generator=g) * 0.1
    inp["c2"] = torch.randn(3, 2, 64, generator=g) * 0.1
    inp["ln_g"] = 1.0 + 0.2 * torch.randn(2, 64, generator=g)
    inp["ln_b"] = 0.1 * torch.randn(2, 64, generator=g)
    got = run_mlp(inp)
    assert int(got["status"].item()) == 0
    compare(got, oracle_mlp(inp), KEYS, TOL["bf16"])


def test_mlp_tc_causality_bit_exact(mlp_form):
    inp = _tc(T=64, B=1, H=2)
    base = run_mlp(inp)
    t = 37
    for key in ("Q", "K", "V"):
        pert = dict(inp)
        pert[key] = inp[key].clone()
        pert[key][0, 1, t] += 0.5
        r = run_mlp(pert)
        assert torch.equal(r["Z"][:, :, :t], base["Z"][:, :, :t]), key
        assert torch.equal(r["loss"][:, :, :t], base["loss"][:, :, :t]), key
        assert torch.equal(r["Z"][:, 0], base["Z"][:, 0]), key
        assert not torch.equal(r["Z"][0, 1, t:], base["Z"][0, 1, t:]), key


def test_mlp_tc_chain_permutation(mlp_form):
    inp = _tc(T=32, B=3, H=2)
    base = run_mlp(inp)
    perm = torch.tensor([2, 0, 1])
    pinp = dict(inp)
    for k in ("Q", "K", "V", "eta"):
        pinp[k] = inp[k][perm].contiguous()
    r = run_mlp(pinp)
    for k in KEYS:
        assert torch.equal(r[k], base[k][perm]), k


def test_mlp_tc_resume_two_calls(mlp_form):
    inp = _tc(T=96, B=1, H=2)
    full = run_mlp(inp)
    T1 = 48
    a, bb = dict(inp), dict(inp)
    for k in ("Q", "K", "V", "eta"):
        a[k] = inp[k][:, :, :T1].contiguous()
        bb[k] = inp[k][:, :, T1:].contiguous()
    ra = run_mlp(a)
    for k in ("W1", "c1", "W2", "c2"):
        bb[k] = ra[k].cpu()
    rb = run_mlp(bb)
    z = torch.cat([ra["Z"], rb["Z"]], 2)
    assert rel_err(to_np(z), to_np(full["Z"])) < 1e-2
    assert rel_err(to_np(rb["W2"]), to_np(full["W2"])) < 1e-2


def test_mlp_tc_outputs_fully_written(mlp_form):
    inp = _tc(T=32, B=2, H=2)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    nan = lambda *s: torch.full(s, float("nan"), device="cuda")
    out = {"Z": nan(2, 2, 32, 64), "W1": nan(2, 2, 256, 64), "c1": nan(2, 2, 256), "W2": nan(2, 2, 64, 256),
           "c2": nan(2, 2, 64), "loss": nan(2, 2, 32), "inner_loss": nan(2, 2, 32)}
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    r = ttt.ttt_mlp_forward(d["Q"], d["K"], d["V"], d["eta"], d["W1"], d["c1"], d["W2"], d["c2"], d["ln_g"],
                            d["ln_b"], mb=16, out=out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for k in out:
        assert torch.isfinite(r[k]).all(), k


def test_mlp_tc_forms_agree():
    """The two-CTA cluster form (hidden units split, partial sums exchanged)
    against the one-CTA form: the same arithmetic up to the order of the sums
    over the hidden units, so they agree far inside the oracle tolerance; each
    form is deterministic."""
    inp = _tc(T=256, B=2, H=3, seed=93)
    try:
        ttt.mlp_cluster_mode(0)
        one = run_mlp(inp)
        ttt.mlp_cluster_mode(2)
        two = run_mlp(inp)
        again = run_mlp(inp)
    finally:
        ttt.mlp_cluster_mode(1)
    assert int(one["status"].item()) == 0 and int(two["status"].item()) == 0
    for k in KEYS:
        assert torch.equal(two[k], again[k]), k
        e = rel_err(to_np(two[k]), to_np(one[k]))
        assert e <= 2e-3, (k, e)


def test_mlp_cluster_mode_default_and_readback():
    assert ttt.mlp_cluster_mode(-1) == 1
    assert ttt.mlp_cluster_mode(7) == 1
    assert ttt.mlp_cluster_mode(0) == 0
    assert ttt.mlp_cluster_mode(1) == 1


@pytest.mark.parametrize("T", [16, 48])
def test_mlp_tc_single_chain(T, mlp_form):
    """One (sequence, head) chain: one CTA, or one cluster of two, on the whole GPU."""
    inp = _tc(T=T, B=1, H=1, seed=97)
    got = run_mlp(inp)
    assert int(got["status"].item()) == 0
    compare(got, oracle_mlp(inp), KEYS, TOL["bf16"])
