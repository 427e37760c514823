"""Mini-batch matrix ("dual") form of the TTT inner loop, fp64 numpy.

TEST INFRASTRUCTURE (see the package docstring). Written independently of the
C token loop in ``ttt_oracle.c``; the pin ``primal == dual`` checks one against
the other.

The "TTT layer" section of the Test-Time Training survey page names a dual form
that does not materialise per-token gradients but prints no formula. The form
below is the plain algebra of the mini-batch rule (Eq. 5 of the End-to-End
Test-Time Training review, section 2.3) with the in-batch prefix output of the
survey's Eq. 5. For mini-batch i with key/query/value rows K, Q, V (b x d),
learning rates eta (b) and anchor (W, c) = (W_{i-1}, c_{i-1}):

    Y  = K W^T + 1 c^T                      f_res of every key at the anchor
    G  = d l_s / d y_s  (rows, through LN)  Eq. 4 gradient w.r.t. f_res output
    A  = tril((Q K^T + 1) * eta^T / b)      A[t, s] = (eta_s / b)(q_t.k_s + 1), s <= t
    Yq = Q W^T + 1 c^T - A G                = W_t q_t + c_t for every t
    Z  = Q + LN(Yq)
    W <- W - (1/b) G^T diag(eta) K,  c <- c - (1/b) G^T eta

For TTT-MLP the same holds per layer: layer 1 sees the keys/queries, layer 2
sees the GELU activations X2 of keys (anchor weights) and queries (prefix
weights).

Output rules: "prefix" is the form above. "anchor" (every prediction of a
mini-batch made with the weights before it, review section 2.3) drops A:
Yq = Q W^T + 1 c^T. "key" (the review's simplified output rule, Eq. 9) is the
anchor rule with the keys as queries, so Yq = Y and Z - V = E.

With ``partial_tail`` the last T % b rows form a shorter batch that uses the
same 1/b and masks but leaves (W, c) at the anchor: it is emitted, not committed.
"""
from __future__ import annotations

import numpy as np

_GELU_A = np.sqrt(2.0 / np.pi)
_GELU_C = 0.044715


def _ln(y, g, bt, eps):
    mu = y.mean(-1, keepdims=True)
    var = ((y - mu) ** 2).mean(-1, keepdims=True)
    rstd = 1.0 / np.sqrt(var + eps)
    yhat = (y - mu) * rstd
    return yhat, rstd, g * yhat + bt


def _ln_bwd(yhat, rstd, g, dout):
    dh = dout * g
    return rstd * (dh - dh.mean(-1, keepdims=True) - yhat * (dh * yhat).mean(-1, keepdims=True))


def _gelu(u):
    return 0.5 * u * (1.0 + np.tanh(_GELU_A * (u + _GELU_C * u ** 3)))


def _gelu_prime(u):
    th = np.tanh(_GELU_A * (u + _GELU_C * u ** 3))
    return 0.5 * (1.0 + th) + 0.5 * u * (1.0 - th * th) * _GELU_A * (1.0 + 3.0 * _GELU_C * u * u)


def _recon(x, y, v, g, bt, eps, ln_res):
    """Rows: E = f(x) - v, loss ||E||^2 and G = d loss / d y."""
    if ln_res:
        yhat, rstd, out = _ln(y, g, bt, eps)
        E = x + out - v
        G = _ln_bwd(yhat, rstd, g, 2.0 * E)
    else:
        E = y - v
        G = 2.0 * E
    return (E * E).sum(-1), G


def _out(x, y, g, bt, eps, ln_res):
    if ln_res:
        return x + _ln(y, g, bt, eps)[2]
    return y


def _broadcast_init(a, B):
    a = np.asarray(a, np.float64)
    return np.broadcast_to(a, (B,) + a.shape[1:]) if a.shape[0] == 1 else a


def _queries(Q, K, rule):
    if rule not in ("prefix", "anchor", "key"):
        raise ValueError(rule)
    return K if rule == "key" else Q


def ttt_linear_dual(Q, K, V, eta, W0, c0, ln_g, ln_b, *, b, eps=1e-6, ln_res=True, rule="prefix",
                    partial_tail=False):
    Q = _queries(Q, K, rule)
    Q, K, V, eta = (np.asarray(a, np.float64) for a in (Q, K, V, eta))
    B, H, T, d = Q.shape
    W0 = _broadcast_init(W0, B)
    c0 = _broadcast_init(c0, B)
    Z = np.empty_like(Q)
    Wf = np.empty((B, H, d, d))
    cf = np.empty((B, H, d))
    loss = np.empty((B, H, T))
    inner = np.empty((B, H, T))
    mask = np.tril(np.ones((b, b))) if rule == "prefix" else np.zeros((b, b))
    for bi in range(B):
        for hi in range(H):
            W = W0[bi, hi].copy()
            c = c0[bi, hi].copy()
            g, bt = np.asarray(ln_g[hi], np.float64), np.asarray(ln_b[hi], np.float64)
            for i in range(-(-T // b) if partial_tail else T // b):
                sl = slice(i * b, min((i + 1) * b, T))
                k, q, v, e = K[bi, hi, sl], Q[bi, hi, sl], V[bi, hi, sl], eta[bi, hi, sl]
                nb = k.shape[0]
                l_in, G = _recon(k, k @ W.T + c, v, g, bt, eps, ln_res)
                A = mask[:nb, :nb] * (q @ k.T + 1.0) * (e / b)[None, :]
                Yq = q @ W.T + c - A @ G
                z = _out(q, Yq, g, bt, eps, ln_res)
                Z[bi, hi, sl] = z
                loss[bi, hi, sl] = ((z - v) ** 2).sum(-1)
                inner[bi, hi, sl] = l_in
                if nb == b:
                    Ge = G * (e / b)[:, None]
                    W = W - Ge.T @ k
                    c = c - Ge.sum(0)
            Wf[bi, hi], cf[bi, hi] = W, c
    return dict(Z=Z, W=Wf, c=cf, loss=loss, inner_loss=inner)


def ttt_mlp_dual(Q, K, V, eta, W1, c1, W2, c2, ln_g, ln_b, *, b, eps=1e-6, ln_res=True, rule="prefix",
                 partial_tail=False):
    Q = _queries(Q, K, rule)
    Q, K, V, eta = (np.asarray(a, np.float64) for a in (Q, K, V, eta))
    B, H, T, d = Q.shape
    W1, c1, W2, c2 = (_broadcast_init(a, B) for a in (W1, c1, W2, c2))
    h = W1.shape[-2]
    Z = np.empty_like(Q)
    out = dict(W1=np.empty((B, H, h, d)), c1=np.empty((B, H, h)),
               W2=np.empty((B, H, d, h)), c2=np.empty((B, H, d)))
    loss = np.empty((B, H, T))
    inner = np.empty((B, H, T))
    mask = np.tril(np.ones((b, b))) if rule == "prefix" else np.zeros((b, b))
    for bi in range(B):
        for hi in range(H):
            w1, b1 = W1[bi, hi].copy(), c1[bi, hi].copy()
            w2, b2 = W2[bi, hi].copy(), c2[bi, hi].copy()
            g, bt = np.asarray(ln_g[hi], np.float64), np.asarray(ln_b[hi], np.float64)
            for i in range(-(-T // b) if partial_tail else T // b):
                sl = slice(i * b, min((i + 1) * b, T))
                k, q, v, e = K[bi, hi, sl], Q[bi, hi, sl], V[bi, hi, sl], eta[bi, hi, sl]
                nb = k.shape[0]
                Z1 = k @ w1.T + b1
                X2 = _gelu(Z1)
                l_in, G = _recon(k, X2 @ w2.T + b2, v, g, bt, eps, ln_res)
                G1 = (G @ w2) * _gelu_prime(Z1)
                A1 = mask[:nb, :nb] * (q @ k.T + 1.0) * (e / b)[None, :]
                Z1q = q @ w1.T + b1 - A1 @ G1
                X2q = _gelu(Z1q)
                A2 = mask[:nb, :nb] * (X2q @ X2.T + 1.0) * (e / b)[None, :]
                Yq = X2q @ w2.T + b2 - A2 @ G
                z = _out(q, Yq, g, bt, eps, ln_res)
                Z[bi, hi, sl] = z
                loss[bi, hi, sl] = ((z - v) ** 2).sum(-1)
                inner[bi, hi, sl] = l_in
                if nb == b:
                    Ge = G * (e / b)[:, None]
                    G1e = G1 * (e / b)[:, None]
                    w2 = w2 - Ge.T @ X2
                    b2 = b2 - Ge.sum(0)
                    w1 = w1 - G1e.T @ k
                    b1 = b1 - G1e.sum(0)
            out["W1"][bi, hi], out["c1"][bi, hi] = w1, b1
            out["W2"][bi, hi], out["c2"][bi, hi] = w2, b2
    return dict(Z=Z, loss=loss, inner_loss=inner, **out)
