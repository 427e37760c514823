"""Gradients of the TTT-Linear inner loop with respect to its inputs, fp64.

TEST INFRASTRUCTURE (see the package docstring): only the test suite,
``__graft_entry__.smoke()`` and the CPU legs of ``bench.py`` use it.

Why a backward pass: the survey page's "TTT layer" section trains the outer
parameters (the projections that make Q, K, V and the learning-rate gate, the
initial weights W_0 and the frozen LayerNorm) by ordinary backpropagation
through the whole inner loop, and that differentiates through every update
W_t = W_{t-1} - (eta_t/b) grad l_t(W_{i-1}): a gradient of a gradient, as
section 2.2 of the "End-to-End Test-Time Training for Long Context" review
points out (the update rule itself contains a gradient). Section 3.7 of the
same review names the resulting training latency as the method's main
limitation.

What is computed: for upstream gradients dZ [B,H,T,d] (and optionally dW_n,
dc_n on the final state) the gradients of

    J = sum(dZ * Z) + sum(dW_n * W_n) + sum(dc_n * c_n)

with respect to Q, K, V, eta (or the gate logits), W0, c0, ln_g and ln_b, for
the prefix output rule (Eq. 5 of the survey's "TTT layer" section) and T a
multiple of b. ``ttt_mlp_backward`` does the same for TTT-MLP (fast weights
W1, c1, W2, c2 of f_res(x) = W2 gelu_tanh(W1 x + c1) + c2).

How: the forward is the primal token loop written once more in plain torch
fp64, not the matrix form, so that it reads like the pages:

* at the start of mini-batch i the anchor (W, c) = (W_{i-1}, c_{i-1});
* every token s of the batch gets its own copy of the anchor, its inner loss
  l_s = || k_s + LN(W k_s + c) - v_s ||^2 (Eq. 4, residual LN form), and
  torch.autograd.grad of l_s with respect to its copy, with create_graph so that
  the gradient itself stays differentiable;
* tokens t = 1..b in order: W_t = W_{t-1} - (eta_t/b) grad l_t(W_{i-1}),
  likewise c (Eq. 2 with the 1/b of the mini-batch rule, review Eq. 5);
  z_t = q_t + LN(W_t q_t + c_t) (survey Eq. 5);
* W_i = W_b.

The outer gradients are then one torch.autograd.grad of J (reverse mode
through both levels). Autograd is the library primitive here; the stated loop
is what it differentiates. The initial weights and LayerNorm parameters are
expanded to one copy per chain before the loop, so their gradients come back
per chain ([B,H,...]); a shared W_0 (or the [H,d] LayerNorm) takes the sum over
the sequences.
"""
from __future__ import annotations

import numpy as np
import torch


def _ln(y, g, bt, eps):
    mu = y.mean(-1, keepdim=True)
    var = ((y - mu) ** 2).mean(-1, keepdim=True)
    return g * (y - mu) / torch.sqrt(var + eps) + bt


def _t(a):
    return torch.as_tensor(np.ascontiguousarray(np.asarray(a, dtype=np.float64)))


def _per_chain(a, B, H, tail):
    """[B|1, H, *tail] or [H, *tail] -> a fresh [B, H, *tail] copy."""
    a = _t(a)
    if a.dim() == 1 + len(tail):  # [H, ...]
        a = a.unsqueeze(0)
    return a.expand(B, H, *tail).clone()


def linear_forward(Q, K, V, eta, W0, c0, ln_g, ln_b, *, b, eps=1e-6, eta_gate=False, eta_base=1.0):
    """Primal token loop in differentiable torch fp64 (prefix rule).

    All arguments are torch fp64 tensors already in per-chain form: Q, K, V
    [B,H,T,d], eta [B,H,T] (gate logits when ``eta_gate``), W0 [B,H,d,d], c0,
    ln_g, ln_b [B,H,d]. Returns Z [B,H,T,d], W_n, c_n."""
    B, H, T, d = Q.shape
    if T % b:
        raise ValueError("T must be a multiple of b")
    lr = eta_base * torch.sigmoid(eta) if eta_gate else eta
    g = ln_g.unsqueeze(2)
    bt = ln_b.unsqueeze(2)
    W, c = W0, c0
    Z = []
    for t0 in range(0, T, b):
        ks, vs, qs = K[:, :, t0:t0 + b], V[:, :, t0:t0 + b], Q[:, :, t0:t0 + b]
        # one copy of the anchor per token: grad l_s(W_{i-1}, c_{i-1}) for each s
        Wk = W.unsqueeze(2).repeat(1, 1, b, 1, 1)
        ck = c.unsqueeze(2).repeat(1, 1, b, 1)
        y = torch.einsum("bhsji,bhsi->bhsj", Wk, ks) + ck
        l = ((ks + _ln(y, g, bt, eps) - vs) ** 2).sum(-1)
        gW, gc = torch.autograd.grad(l.sum(), (Wk, ck), create_graph=True)
        for s in range(b):
            e = (lr[:, :, t0 + s] / b)
            W = W - e[:, :, None, None] * gW[:, :, s]
            c = c - e[:, :, None] * gc[:, :, s]
            yq = torch.einsum("bhji,bhi->bhj", W, qs[:, :, s]) + c
            Z.append(qs[:, :, s] + _ln(yq, ln_g, ln_b, eps))
    return torch.stack(Z, dim=2), W, c


_GELU_A = (2.0 / np.pi) ** 0.5
_GELU_C = 0.044715


def _gelu(u):
    return 0.5 * u * (1.0 + torch.tanh(_GELU_A * (u + _GELU_C * u ** 3)))


def mlp_forward(Q, K, V, eta, W1, c1, W2, c2, ln_g, ln_b, *, b, eps=1e-6, eta_gate=False, eta_base=1.0):
    """TTT-MLP primal token loop in differentiable torch fp64 (prefix rule):
    f_res(x) = W2 gelu_tanh(W1 x + c1) + c2, the same steps as ``linear_forward``
    with the four fast weights. W1 [B,H,h,d], c1 [B,H,h], W2 [B,H,d,h], c2, ln_g,
    ln_b [B,H,d]. Returns Z and the final (W1, c1, W2, c2)."""
    B, H, T, d = Q.shape
    if T % b:
        raise ValueError("T must be a multiple of b")
    lr = eta_base * torch.sigmoid(eta) if eta_gate else eta
    g = ln_g.unsqueeze(2)
    bt = ln_b.unsqueeze(2)
    st = [W1, c1, W2, c2]
    Z = []

    def f_res(w1, a1, w2, a2, x, sub):
        # x [..., d]; weights with an extra per-token axis when ``sub`` ("bhs")
        if sub:
            h1 = torch.einsum("bhsnd,bhsd->bhsn", w1, x) + a1
            return torch.einsum("bhsdn,bhsn->bhsd", w2, _gelu(h1)) + a2
        h1 = torch.einsum("bhnd,bhd->bhn", w1, x) + a1
        return torch.einsum("bhdn,bhn->bhd", w2, _gelu(h1)) + a2

    for t0 in range(0, T, b):
        ks, vs, qs = K[:, :, t0:t0 + b], V[:, :, t0:t0 + b], Q[:, :, t0:t0 + b]
        # one copy of the anchor per token: grad l_s(W_{i-1}) for each token s
        cp = [w.unsqueeze(2).repeat(1, 1, b, *([1] * (w.dim() - 2))) for w in st]
        y = f_res(*cp, ks, True)
        l = ((ks + _ln(y, g, bt, eps) - vs) ** 2).sum(-1)
        grads = torch.autograd.grad(l.sum(), cp, create_graph=True)
        cur = list(st)
        for s in range(b):
            e = lr[:, :, t0 + s] / b
            cur = [w - e.reshape(B, H, *([1] * (w.dim() - 2))) * gr[:, :, s] for w, gr in zip(cur, grads)]
            Z.append(qs[:, :, s] + _ln(f_res(*cur, qs[:, :, s], False), ln_g, ln_b, eps))
        st = cur
    return torch.stack(Z, dim=2), st


def ttt_mlp_backward(Q, K, V, eta, W1, c1, W2, c2, ln_g, ln_b, dZ, dW1_n=None, dc1_n=None, dW2_n=None,
                     dc2_n=None, *, b, eps=1e-6, eta_gate=False, eta_base=1.0):
    """Outer gradients of the TTT-MLP inner loop (see the module docstring).

    Inputs as for ``oracle.ttt_mlp`` (W1 [B|1,H,h,d], c1 [B|1,H,h], W2 [B|1,H,d,h],
    c2 [B|1,H,d], ln_g, ln_b [H,d]) plus dZ [B,H,T,d] and optional final-state
    seeds. Returns numpy fp64 dQ, dK, dV, deta and per chain dW1, dc1, dW2, dc2,
    dln_g, dln_b; also Z and the final state of the forward."""
    Qt, Kt, Vt, et = (_t(a) for a in (Q, K, V, eta))
    B, H, T, d = Qt.shape
    h = np.asarray(W1).shape[-2]
    W1t = _per_chain(W1, B, H, (h, d))
    c1t = _per_chain(c1, B, H, (h,))
    W2t = _per_chain(W2, B, H, (d, h))
    c2t = _per_chain(c2, B, H, (d,))
    gt = _per_chain(ln_g, B, H, (d,))
    btt = _per_chain(ln_b, B, H, (d,))
    leaves = [Qt, Kt, Vt, et, W1t, c1t, W2t, c2t, gt, btt]
    for a in leaves:
        a.requires_grad_(True)
    with torch.enable_grad():
        Z, fin = mlp_forward(Qt, Kt, Vt, et, W1t, c1t, W2t, c2t, gt, btt, b=b, eps=eps, eta_gate=eta_gate,
                             eta_base=eta_base)
        J = (Z * _t(dZ)).sum()
        for w, sd in zip(fin, (dW1_n, dc1_n, dW2_n, dc2_n)):
            if sd is not None:
                J = J + (w * _t(sd)).sum()
        grads = torch.autograd.grad(J, leaves, allow_unused=True)
    names = ["dQ", "dK", "dV", "deta", "dW1", "dc1", "dW2", "dc2", "dln_g", "dln_b"]
    out = {n: (torch.zeros_like(leaf) if gr is None else gr).detach().numpy()
           for n, gr, leaf in zip(names, grads, leaves)}
    out["Z"] = Z.detach().numpy()
    for n, w in zip(("W1", "c1", "W2", "c2"), fin):
        out[n] = w.detach().numpy()
    return out


def ttt_linear_backward(Q, K, V, eta, W0, c0, ln_g, ln_b, dZ, dW_n=None, dc_n=None, *, b, eps=1e-6,
                        eta_gate=False, eta_base=1.0):
    """Outer gradients of the TTT-Linear inner loop (see the module docstring).

    Inputs as for ``oracle.ttt_linear`` (W0 [B|1,H,d,d], c0 [B|1,H,d], ln_g,
    ln_b [H,d]) plus dZ [B,H,T,d] and the optional final-state seeds dW_n
    [B,H,d,d], dc_n [B,H,d]. Returns numpy fp64 arrays dQ, dK, dV, deta
    (w.r.t. the gate logits when ``eta_gate``) [B,H,T(,d)], and per chain dW0
    [B,H,d,d], dc0, dln_g, dln_b [B,H,d]; also Z, W and c of the forward."""
    Qt, Kt, Vt, et = (_t(a) for a in (Q, K, V, eta))
    B, H, T, d = Qt.shape
    W0t = _per_chain(W0, B, H, (d, d))
    c0t = _per_chain(c0, B, H, (d,))
    gt = _per_chain(ln_g, B, H, (d,))
    btt = _per_chain(ln_b, B, H, (d,))
    leaves = [Qt, Kt, Vt, et, W0t, c0t, gt, btt]
    for a in leaves:
        a.requires_grad_(True)
    with torch.enable_grad():
        Z, Wn, cn = linear_forward(Qt, Kt, Vt, et, W0t, c0t, gt, btt, b=b, eps=eps, eta_gate=eta_gate,
                                   eta_base=eta_base)
        J = (Z * _t(dZ)).sum()
        if dW_n is not None:
            J = J + (Wn * _t(dW_n)).sum()
        if dc_n is not None:
            J = J + (cn * _t(dc_n)).sum()
        grads = torch.autograd.grad(J, leaves, allow_unused=True)
    names = ["dQ", "dK", "dV", "deta", "dW0", "dc0", "dln_g", "dln_b"]
    out = {}
    for n, gr, leaf in zip(names, grads, leaves):
        out[n] = (torch.zeros_like(leaf) if gr is None else gr).detach().numpy()
    out["Z"] = Z.detach().numpy()
    out["W"] = Wn.detach().numpy()
    out["c"] = cn.detach().numpy()
    return out
