"""Pins of the fp64 backward oracle (``oracle.backward``) against things other than itself.

* central finite differences of J = sum(dZ*Z) + sum(dW_n*W_n) + sum(dc_n*c_n)
  computed with the C primal token loop (``oracle.ttt_linear``, separate code
  that is pinned on its own), along a random direction of every input: a
  dropped second-order term, a wrong sign or a transposed operand in the
  backward moves the directional derivative far beyond the fp64 difference
  error;
* eta = 0 (no update): the keys and values drop out (dK = dV = 0 exactly) and
  the rest is the gradient of q + LN(W_0 q + c_0) through the library LayerNorm;
* the forward inside the backward oracle reproduces the C oracle's Z and final
  state.

The same three pins hold ``ttt_mlp_backward`` (TTT-MLP) against ``oracle.ttt_mlp``,
with the eta = 0 case against the library LayerNorm and tanh-GELU.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle.backward import ttt_linear_backward, ttt_mlp_backward

INPUTS = ["Q", "K", "V", "eta", "W0", "c0", "ln_g", "ln_b"]


def _case(rng, B=2, H=2, T=12, d=5, shared=True, gate=False):
    Q, K, V = (rng.standard_normal((B, H, T, d)) for _ in range(3))
    eta = rng.standard_normal((B, H, T)) if gate else rng.uniform(0.2, 1.0, (B, H, T))
    lead = 1 if shared else B
    x = dict(Q=Q, K=K, V=V, eta=eta, W0=rng.standard_normal((lead, H, d, d)) * 0.3,
             c0=rng.standard_normal((lead, H, d)) * 0.3, ln_g=rng.uniform(0.6, 1.4, (H, d)),
             ln_b=rng.standard_normal((H, d)) * 0.1)
    seeds = dict(dZ=rng.standard_normal((B, H, T, d)), dW_n=rng.standard_normal((B, H, d, d)),
                 dc_n=rng.standard_normal((B, H, d)))
    return x, seeds


def _J(x, seeds, b, gate):
    r = oracle.ttt_linear(x["Q"], x["K"], x["V"], x["eta"], x["W0"], x["c0"], x["ln_g"], x["ln_b"], b=b,
                          eta_gate=gate, eta_base=0.8)
    return (r["Z"] * seeds["dZ"]).sum() + (r["W"] * seeds["dW_n"]).sum() + (r["c"] * seeds["dc_n"]).sum()


def _directional(grad, name, x):
    """<grad, D> for the per-chain gradient of an input that may be shared over B."""
    if name in ("ln_g", "ln_b"):
        return grad.sum(0)
    if name in ("W0", "c0", "W1", "c1", "W2", "c2") and x[name].shape[0] == 1:
        return grad.sum(0, keepdims=True)
    return grad


@pytest.mark.parametrize("b,shared,gate", [(4, True, False), (1, False, False), (12, True, False),
                                           (4, False, True)])
def test_backward_oracle_matches_finite_differences(b, shared, gate):
    rng = np.random.default_rng(11 + b + 2 * shared + 5 * gate)
    x, seeds = _case(rng, shared=shared, gate=gate)
    out = ttt_linear_backward(*(x[n] for n in INPUTS), seeds["dZ"], seeds["dW_n"], seeds["dc_n"], b=b,
                              eta_gate=gate, eta_base=0.8)
    h = 1e-6
    for name in INPUTS:
        D = rng.standard_normal(x[name].shape)
        xp, xm = dict(x), dict(x)
        xp[name] = x[name] + h * D
        xm[name] = x[name] - h * D
        fd = (_J(xp, seeds, b, gate) - _J(xm, seeds, b, gate)) / (2 * h)
        an = float((_directional(out["d" + name], name, x) * D).sum())
        assert abs(fd - an) <= 1e-7 * max(1.0, abs(fd)), (name, fd, an)


def test_backward_oracle_forward_matches_c_oracle():
    rng = np.random.default_rng(5)
    x, seeds = _case(rng, T=16)
    out = ttt_linear_backward(*(x[n] for n in INPUTS), seeds["dZ"], b=8)
    ref = oracle.ttt_linear(*(x[n] for n in INPUTS), b=8)
    for k in ("Z", "W", "c"):
        np.testing.assert_allclose(out[k], ref[k], rtol=0, atol=1e-12)


def test_backward_oracle_without_updates_is_a_layer_norm_gradient():
    rng = np.random.default_rng(6)
    x, seeds = _case(rng, B=1, H=2, T=8, d=6, shared=False)
    x["eta"] = np.zeros_like(x["eta"])
    out = ttt_linear_backward(*(x[n] for n in INPUTS), seeds["dZ"], seeds["dW_n"], seeds["dc_n"], b=4)
    assert not out["dK"].any() and not out["dV"].any()
    Q = torch.tensor(x["Q"], requires_grad=True)
    W0 = torch.tensor(x["W0"], requires_grad=True)
    c0 = torch.tensor(x["c0"], requires_grad=True)
    g = torch.tensor(x["ln_g"], requires_grad=True)
    bt = torch.tensor(x["ln_b"], requires_grad=True)
    y = torch.einsum("bhji,bhti->bhtj", W0, Q) + c0[:, :, None, :]
    d = y.shape[-1]
    z = torch.stack([Q[:, h] + F.layer_norm(y[:, h], (d,), g[h], bt[h], eps=1e-6) for h in range(2)], 1)
    J = (z * torch.tensor(seeds["dZ"])).sum() + (W0 * torch.tensor(seeds["dW_n"])).sum() \
        + (c0 * torch.tensor(seeds["dc_n"])).sum()
    gQ, gW, gc, gg, gb = torch.autograd.grad(J, (Q, W0, c0, g, bt))
    np.testing.assert_allclose(out["dQ"], gQ.numpy(), rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(out["dW0"], gW.numpy(), rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(out["dc0"], gc.numpy(), rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(out["dln_g"].sum(0), gg.numpy(), rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(out["dln_b"].sum(0), gb.numpy(), rtol=1e-10, atol=1e-10)


MLP_INPUTS = ["Q", "K", "V", "eta", "W1", "c1", "W2", "c2", "ln_g", "ln_b"]


def _mlp_case(rng, B=1, H=2, T=12, d=4, h=6, shared=True, gate=False):
    Q, K, V = (rng.standard_normal((B, H, T, d)) for _ in range(3))
    eta = rng.standard_normal((B, H, T)) if gate else rng.uniform(0.2, 1.0, (B, H, T))
    lead = 1 if shared else B
    x = dict(Q=Q, K=K, V=V, eta=eta, W1=rng.standard_normal((lead, H, h, d)) * 0.4,
             c1=rng.standard_normal((lead, H, h)) * 0.2, W2=rng.standard_normal((lead, H, d, h)) * 0.4,
             c2=rng.standard_normal((lead, H, d)) * 0.2, ln_g=rng.uniform(0.6, 1.4, (H, d)),
             ln_b=rng.standard_normal((H, d)) * 0.1)
    seeds = dict(dZ=rng.standard_normal((B, H, T, d)), dW1_n=rng.standard_normal((B, H, h, d)),
                 dc1_n=rng.standard_normal((B, H, h)), dW2_n=rng.standard_normal((B, H, d, h)),
                 dc2_n=rng.standard_normal((B, H, d)))
    return x, seeds


def _J_mlp(x, seeds, b, gate):
    r = oracle.ttt_mlp(*(x[n] for n in MLP_INPUTS), b=b, eta_gate=gate, eta_base=0.8)
    return (r["Z"] * seeds["dZ"]).sum() + sum((r[k] * seeds["d%s_n" % k]).sum() for k in ("W1", "c1", "W2", "c2"))


@pytest.mark.parametrize("b,shared,gate", [(4, True, False), (1, False, False), (12, True, True)])
def test_mlp_backward_oracle_matches_finite_differences(b, shared, gate):
    rng = np.random.default_rng(21 + b + 2 * shared + 5 * gate)
    x, seeds = _mlp_case(rng, shared=shared, gate=gate)
    out = ttt_mlp_backward(*(x[n] for n in MLP_INPUTS), seeds["dZ"], seeds["dW1_n"], seeds["dc1_n"],
                           seeds["dW2_n"], seeds["dc2_n"], b=b, eta_gate=gate, eta_base=0.8)
    h = 1e-6
    for name in MLP_INPUTS:
        D = rng.standard_normal(x[name].shape)
        xp, xm = dict(x), dict(x)
        xp[name] = x[name] + h * D
        xm[name] = x[name] - h * D
        fd = (_J_mlp(xp, seeds, b, gate) - _J_mlp(xm, seeds, b, gate)) / (2 * h)
        an = float((_directional(out["d" + name], name, x) * D).sum())
        assert abs(fd - an) <= 1e-7 * max(1.0, abs(fd)), (name, fd, an)


def test_mlp_backward_oracle_forward_matches_c_oracle():
    rng = np.random.default_rng(22)
    x, seeds = _mlp_case(rng, T=16)
    out = ttt_mlp_backward(*(x[n] for n in MLP_INPUTS), seeds["dZ"], b=8)
    ref = oracle.ttt_mlp(*(x[n] for n in MLP_INPUTS), b=8)
    for k in ("Z", "W1", "c1", "W2", "c2"):
        np.testing.assert_allclose(out[k], ref[k], rtol=0, atol=1e-12)


def test_mlp_backward_oracle_without_updates_is_a_library_gradient():
    rng = np.random.default_rng(23)
    x, seeds = _mlp_case(rng, B=1, H=2, T=8, d=5, h=7, shared=False)
    x["eta"] = np.zeros_like(x["eta"])
    out = ttt_mlp_backward(*(x[n] for n in MLP_INPUTS), seeds["dZ"], b=4)
    assert not out["dK"].any() and not out["dV"].any()
    t = {k: torch.tensor(x[k], requires_grad=True) for k in ("Q", "W1", "c1", "W2", "c2", "ln_g", "ln_b")}
    h1 = torch.einsum("bhnd,bhtd->bhtn", t["W1"], t["Q"]) + t["c1"][:, :, None, :]
    y = torch.einsum("bhdn,bhtn->bhtd", t["W2"], F.gelu(h1, approximate="tanh")) + t["c2"][:, :, None, :]
    d = y.shape[-1]
    z = torch.stack([t["Q"][:, i] + F.layer_norm(y[:, i], (d,), t["ln_g"][i], t["ln_b"][i], eps=1e-6)
                     for i in range(2)], 1)
    grads = torch.autograd.grad((z * torch.tensor(seeds["dZ"])).sum(), [t[k] for k in t])
    for k, g in zip(t, grads):
        got = out["d" + k].sum(0) if k in ("ln_g", "ln_b") else out["d" + k]
        np.testing.assert_allclose(got, g.numpy(), rtol=1e-10, atol=1e-10, err_msg=k)
