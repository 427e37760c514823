"""Pins of the fp64 oracle against things other than itself.

Each check is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign, a transposed operand, the wrong in-batch rule, a missing 1/b) fails
at least one of them:

* golden: a worked example derived by hand (tests/golden/linear_noln_d2.txt);
* closed form: gradient of ||W k + c - v||^2 is 2(Wk + c - v) k^T;
* finite differences and fp64 torch autograd for the LayerNorm/GELU gradients;
* library routines: torch layer_norm and tanh-GELU for the eta = 0 output;
* the per-token listing of Eqs. 2/4/5 of the survey page with autograd
  gradients (b = 1), and its mini-batch form (Eq. 5 of the E2E review);
* Theorem 1 of the survey's "relation to attention" section: linear f, batch
  GD, eta = 1/2, W_0 = 0 gives causal linear attention;
* invariants: LayerNorm row statistics, causality, resume, rank of an update;
* primal token loop (C) == dual matrix form (numpy).
"""
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import dual

GOLD = os.path.join(os.path.dirname(__file__), "golden", "linear_noln_d2.txt")


def _rand_linear(rng, B=2, H=2, T=32, d=8, shared=True, wscale=0.3):
    Q, K, V = (rng.standard_normal((B, H, T, d)) for _ in range(3))
    eta = rng.uniform(0.2, 0.8, (B, H, T))
    lead = 1 if shared else B
    W0 = rng.standard_normal((lead, H, d, d)) * wscale
    c0 = rng.standard_normal((lead, H, d)) * 0.1
    g = rng.uniform(0.5, 1.5, (H, d))
    bt = rng.standard_normal((H, d)) * 0.1
    return Q, K, V, eta, W0, c0, g, bt


def _rand_mlp(rng, B=1, H=2, T=16, d=6, h=12):
    Q, K, V = (rng.standard_normal((B, H, T, d)) for _ in range(3))
    eta = rng.uniform(0.2, 0.8, (B, H, T))
    W1 = rng.standard_normal((1, H, h, d)) * 0.4
    c1 = rng.standard_normal((1, H, h)) * 0.1
    W2 = rng.standard_normal((1, H, d, h)) * 0.4
    c2 = rng.standard_normal((1, H, d)) * 0.1
    g = rng.uniform(0.5, 1.5, (H, d))
    bt = rng.standard_normal((H, d)) * 0.1
    return Q, K, V, eta, W1, c1, W2, c2, g, bt


# ---------------------------------------------------------------- golden


def _read_golden():
    cases = {}
    for line in open(GOLD):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        case, field, *vals = line.split()
        cases.setdefault(case, {})[field] = np.array([float(v) for v in vals])
    return cases


@pytest.mark.parametrize("b", [1, 2])
def test_golden_hand_example(b):
    gold = _read_golden()["b%d" % b]
    K = np.array([[1.0, 0.0], [0.0, 1.0]])[None, None]
    V = np.array([[1.0, 2.0], [3.0, -1.0]])[None, None]
    Q = np.array([[0.0, 1.0], [1.0, 1.0]])[None, None]
    eta = np.array([0.5, 0.25])[None, None]
    W0 = np.zeros((1, 1, 2, 2))
    c0 = np.zeros((1, 1, 2))
    g, bt = np.ones((1, 2)), np.zeros((1, 2))
    for impl in (oracle.ttt_linear, dual.ttt_linear_dual):
        r = impl(Q, K, V, eta, W0, c0, g, bt, b=b, ln_res=False)
        for f in ("Z", "W", "c", "loss", "inner_loss"):
            np.testing.assert_array_equal(r[f].ravel(), gold[f], err_msg=f)


# ---------------------------------------------------------------- gradients


def test_gradient_closed_form_without_ln():
    rng = np.random.default_rng(2)
    for d in (1, 3, 8):
        W = rng.standard_normal((d, d))
        c = rng.standard_normal(d)
        k, v = rng.standard_normal(d), rng.standard_normal(d)
        l, dW, dc = oracle.linear_token_grad(W, c, k, v, np.ones(d), np.zeros(d), ln_res=False)
        r = W @ k + c - v
        assert l == pytest.approx(float(r @ r), rel=1e-14)
        np.testing.assert_allclose(dW, 2.0 * np.outer(r, k), rtol=1e-14, atol=1e-14)
        np.testing.assert_allclose(dc, 2.0 * r, rtol=1e-14, atol=1e-14)


def _fd_linear(W, c, k, v, g, bt, ln_res, h=1e-6):
    d = k.shape[0]
    dW = np.zeros((d, d))
    dc = np.zeros(d)
    f = lambda W_, c_: oracle.linear_token_grad(W_, c_, k, v, g, bt, ln_res=ln_res)[0]
    for i in range(d):
        for j in range(d):
            Wp, Wm = W.copy(), W.copy()
            Wp[i, j] += h
            Wm[i, j] -= h
            dW[i, j] = (f(Wp, c) - f(Wm, c)) / (2 * h)
        cp, cm = c.copy(), c.copy()
        cp[i] += h
        cm[i] -= h
        dc[i] = (f(W, cp) - f(W, cm)) / (2 * h)
    return dW, dc


@pytest.mark.parametrize("ln_res", [False, True])
def test_gradient_finite_differences(ln_res):
    rng = np.random.default_rng(3)
    for d in (2, 5, 8):
        W = rng.standard_normal((d, d)) * 0.7
        c = rng.standard_normal(d) * 0.3
        k, v = rng.standard_normal(d), rng.standard_normal(d)
        g, bt = rng.uniform(0.5, 1.5, d), rng.standard_normal(d) * 0.2
        _, dW, dc = oracle.linear_token_grad(W, c, k, v, g, bt, ln_res=ln_res)
        fW, fc = _fd_linear(W, c, k, v, g, bt, ln_res)
        scale = max(np.abs(dW).max(), 1.0)
        assert np.abs(dW - fW).max() <= 1e-7 * scale
        assert np.abs(dc - fc).max() <= 1e-7 * scale


def _torch_f_linear(W, c, x, g, bt, eps, ln_res):
    y = W @ x + c
    if not ln_res:
        return y
    return x + F.layer_norm(y, (y.shape[-1],), weight=g, bias=bt, eps=eps)


def _torch_f_mlp(W1, c1, W2, c2, x, g, bt, eps, ln_res):
    y = W2 @ F.gelu(W1 @ x + c1, approximate="tanh") + c2
    if not ln_res:
        return y
    return x + F.layer_norm(y, (y.shape[-1],), weight=g, bias=bt, eps=eps)


def test_gradient_vs_autograd_linear_ln():
    rng = np.random.default_rng(4)
    d = 16
    for _ in range(5):
        W = rng.standard_normal((d, d)) * 0.3
        c = rng.standard_normal(d) * 0.1
        k, v = rng.standard_normal(d), rng.standard_normal(d)
        g, bt = rng.uniform(0.5, 1.5, d), rng.standard_normal(d) * 0.2
        l, dW, dc = oracle.linear_token_grad(W, c, k, v, g, bt)
        Wt = torch.tensor(W, requires_grad=True)
        ct = torch.tensor(c, requires_grad=True)
        lt = (_torch_f_linear(Wt, ct, torch.tensor(k), torch.tensor(g), torch.tensor(bt), 1e-6, True)
              - torch.tensor(v)).pow(2).sum()
        gW, gc = torch.autograd.grad(lt, (Wt, ct))
        assert l == pytest.approx(lt.item(), rel=1e-12)
        np.testing.assert_allclose(dW, gW.numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(dc, gc.numpy(), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("ln_res", [False, True])
def test_gradient_vs_autograd_mlp(ln_res):
    rng = np.random.default_rng(5)
    d, h = 8, 32
    W1 = rng.standard_normal((h, d)) * 0.4
    c1 = rng.standard_normal(h) * 0.2
    W2 = rng.standard_normal((d, h)) * 0.3
    c2 = rng.standard_normal(d) * 0.1
    k, v = rng.standard_normal(d), rng.standard_normal(d)
    g, bt = rng.uniform(0.5, 1.5, d), rng.standard_normal(d) * 0.2
    l, dW1, dc1, dW2, dc2 = oracle.mlp_token_grad(W1, c1, W2, c2, k, v, g, bt, ln_res=ln_res)
    ts = [torch.tensor(a, requires_grad=True) for a in (W1, c1, W2, c2)]
    lt = (_torch_f_mlp(*ts, torch.tensor(k), torch.tensor(g), torch.tensor(bt), 1e-6, ln_res)
          - torch.tensor(v)).pow(2).sum()
    grads = torch.autograd.grad(lt, ts)
    assert l == pytest.approx(lt.item(), rel=1e-12)
    for mine, ref in zip((dW1, dc1, dW2, dc2), grads):
        np.testing.assert_allclose(mine, ref.numpy(), rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- eta = 0


def test_eta_zero_is_library_layernorm_linear():
    rng = np.random.default_rng(6)
    Q, K, V, eta, W0, c0, g, bt = _rand_linear(rng, shared=False)
    eta[:] = 0.0
    r = oracle.ttt_linear(Q, K, V, eta, W0, c0, g, bt, b=8)
    np.testing.assert_array_equal(r["W"], W0)
    np.testing.assert_array_equal(r["c"], c0)
    Qt = torch.tensor(Q)
    y = torch.einsum("bhij,bhtj->bhti", torch.tensor(W0), Qt) + torch.tensor(c0)[:, :, None, :]
    for hh in range(Q.shape[1]):
        ref = Qt[:, hh] + F.layer_norm(y[:, hh], (Q.shape[-1],), weight=torch.tensor(g[hh]),
                                       bias=torch.tensor(bt[hh]), eps=1e-6)
        np.testing.assert_allclose(r["Z"][:, hh], ref.numpy(), rtol=0, atol=1e-12)


def test_eta_zero_is_library_gelu_layernorm_mlp():
    rng = np.random.default_rng(7)
    Q, K, V, eta, W1, c1, W2, c2, g, bt = _rand_mlp(rng)
    eta[:] = 0.0
    r = oracle.ttt_mlp(Q, K, V, eta, W1, c1, W2, c2, g, bt, b=4)
    np.testing.assert_array_equal(r["W1"][0], W1[0])
    np.testing.assert_array_equal(r["W2"][0], W2[0])
    for hh in range(Q.shape[1]):
        q = torch.tensor(Q[0, hh])
        y = F.gelu(q @ torch.tensor(W1[0, hh]).T + torch.tensor(c1[0, hh]), approximate="tanh")
        y = y @ torch.tensor(W2[0, hh]).T + torch.tensor(c2[0, hh])
        ref = q + F.layer_norm(y, (y.shape[-1],), weight=torch.tensor(g[hh]),
                               bias=torch.tensor(bt[hh]), eps=1e-6)
        np.testing.assert_allclose(r["Z"][0, hh], ref.numpy(), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- listings with autograd


def _listing_minibatch(Q, K, V, eta, W0, c0, g, bt, b, mlp=False):
    """Eqs. 2/4/5 of the survey's "TTT layer" section, mini-batched as in Eq. 5 of
    the E2E review, with gradients from torch autograd (not the oracle's hand
    derivation). One chain; returns Z, final weights."""
    T, d = Q.shape
    g, bt = torch.tensor(g), torch.tensor(bt)
    Ws = [torch.tensor(a).clone() for a in W0]
    Z = np.empty((T, d))
    f = _torch_f_mlp if mlp else _torch_f_linear
    for i in range(T // b):
        anchor = [w.clone().requires_grad_(True) for w in Ws]
        grads = []
        for s in range(i * b, (i + 1) * b):
            l = (f(*anchor, torch.tensor(K[s]), g, bt, 1e-6, True) - torch.tensor(V[s])).pow(2).sum()
            grads.append(torch.autograd.grad(l, anchor))
        for j, s in enumerate(range(i * b, (i + 1) * b)):
            Ws = [w - (eta[s] / b) * gr for w, gr in zip(Ws, grads[j])]
            with torch.no_grad():
                Z[s] = f(*Ws, torch.tensor(Q[s]), g, bt, 1e-6, True).numpy()
    return Z, [w.detach().numpy() for w in Ws]


@pytest.mark.parametrize("b", [1, 4])
def test_listing_with_autograd_linear(b):
    rng = np.random.default_rng(8)
    Q, K, V, eta, W0, c0, g, bt = _rand_linear(rng, B=1, H=1, T=16, d=6)
    r = oracle.ttt_linear(Q, K, V, eta, W0, c0, g, bt, b=b)
    Z, (W, c) = _listing_minibatch(Q[0, 0], K[0, 0], V[0, 0], eta[0, 0], (W0[0, 0], c0[0, 0]),
                                   None, g[0], bt[0], b)
    np.testing.assert_allclose(r["Z"][0, 0], Z, rtol=0, atol=1e-11)
    np.testing.assert_allclose(r["W"][0, 0], W, rtol=0, atol=1e-11)
    np.testing.assert_allclose(r["c"][0, 0], c, rtol=0, atol=1e-11)


def _listing_minibatch_mlp(Q, K, V, eta, Ws0, g, bt, b):
    return _listing_minibatch(Q, K, V, eta, Ws0, None, g, bt, b, mlp=True)


@pytest.mark.parametrize("b", [1, 4])
def test_listing_with_autograd_mlp(b):
    rng = np.random.default_rng(9)
    Q, K, V, eta, W1, c1, W2, c2, g, bt = _rand_mlp(rng, H=1, T=12, d=5, h=10)
    r = oracle.ttt_mlp(Q, K, V, eta, W1, c1, W2, c2, g, bt, b=b)
    Z, (w1, b1, w2, b2) = _listing_minibatch_mlp(
        Q[0, 0], K[0, 0], V[0, 0], eta[0, 0], (W1[0, 0], c1[0, 0], W2[0, 0], c2[0, 0]), g[0], bt[0], b)
    np.testing.assert_allclose(r["Z"][0, 0], Z, rtol=0, atol=1e-11)
    for mine, ref in zip((r["W1"], r["c1"], r["W2"], r["c2"]), (w1, b1, w2, b2)):
        np.testing.assert_allclose(mine[0, 0], ref, rtol=0, atol=1e-11)


# ---------------------------------------------------------------- Theorem 1


@pytest.mark.parametrize("T", [1, 7, 24])
def test_theorem1_causal_linear_attention(T):
    """Linear f (no LN/residual), one mini-batch (batch GD at W_0 = 0), step 1/2:
    z_t = sum_{s<=t} v_s (k_s . q_t + 1) -- causal linear attention on keys
    augmented with a constant 1 for the bias c (c_0 = 0)."""
    rng = np.random.default_rng(10)
    d = 5
    Q, K, V = (rng.standard_normal((1, 1, T, d)) for _ in range(3))
    eta = np.full((1, 1, T), T / 2.0)  # eta_t / b = 1/2
    r = oracle.ttt_linear(Q, K, V, eta, np.zeros((1, 1, d, d)), np.zeros((1, 1, d)),
                          np.ones((1, d)), np.zeros((1, d)), b=T, ln_res=False)
    q, k, v = Q[0, 0], K[0, 0], V[0, 0]
    scores = np.tril(q @ k.T + 1.0)          # [t, s], s <= t
    np.testing.assert_allclose(r["Z"][0, 0], scores @ v, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(r["W"][0, 0], v.T @ k, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(r["c"][0, 0], v.sum(0), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- primal == dual


@pytest.mark.parametrize("b", [1, 2, 4, 16])
@pytest.mark.parametrize("ln_res", [True, False])
def test_primal_equals_dual_linear(b, ln_res):
    rng = np.random.default_rng(11 + b)
    args = _rand_linear(rng, T=32, d=8, shared=(b % 2 == 0))
    p = oracle.ttt_linear(*args, b=b, ln_res=ln_res)
    q = dual.ttt_linear_dual(*args, b=b, ln_res=ln_res)
    for f in p:
        scale = max(np.abs(p[f]).max(), 1.0)
        assert np.abs(p[f] - q[f]).max() <= 1e-12 * scale, f


@pytest.mark.parametrize("b", [1, 4, 8])
def test_primal_equals_dual_mlp(b):
    rng = np.random.default_rng(21 + b)
    args = _rand_mlp(rng, B=2, T=16)
    p = oracle.ttt_mlp(*args, b=b)
    q = dual.ttt_mlp_dual(*args, b=b)
    for f in p:
        scale = max(np.abs(p[f]).max(), 1.0)
        assert np.abs(p[f] - q[f]).max() <= 1e-12 * scale, f


# ---------------------------------------------------------------- invariants


def test_layernorm_row_statistics():
    rng = np.random.default_rng(12)
    Q, K, V, eta, W0, c0, g, bt = _rand_linear(rng, T=64, d=16)
    g[:] = 1.0
    bt[:] = 0.0
    r = oracle.ttt_linear(Q, K, V, eta, W0, c0, g, bt, b=16)
    D = r["Z"] - Q
    np.testing.assert_allclose(D.mean(-1), 0.0, atol=1e-12)
    ms = (D ** 2).mean(-1)
    assert np.all(ms < 1.0) and np.all(ms > 0.99)


def test_causality_bit_exact():
    rng = np.random.default_rng(13)
    args = list(_rand_linear(rng, B=1, H=1, T=48, d=8))
    base = oracle.ttt_linear(*args, b=8)
    t = 27
    for idx in (0, 1, 2):
        pert = [a.copy() for a in args]
        pert[idx][0, 0, t] += 0.5
        r = oracle.ttt_linear(*pert, b=8)
        np.testing.assert_array_equal(r["Z"][0, 0, :t], base["Z"][0, 0, :t])
        np.testing.assert_array_equal(r["loss"][0, 0, :t], base["loss"][0, 0, :t])
        assert np.abs(r["Z"][0, 0, t:] - base["Z"][0, 0, t:]).max() > 0


def test_resume_equals_single_call():
    rng = np.random.default_rng(14)
    Q, K, V, eta, W0, c0, g, bt = _rand_linear(rng, T=48, d=8)
    full = oracle.ttt_linear(Q, K, V, eta, W0, c0, g, bt, b=8)
    T1 = 24
    a = oracle.ttt_linear(Q[:, :, :T1], K[:, :, :T1], V[:, :, :T1], eta[:, :, :T1], W0, c0, g, bt, b=8)
    bb = oracle.ttt_linear(Q[:, :, T1:], K[:, :, T1:], V[:, :, T1:], eta[:, :, T1:], a["W"], a["c"],
                           g, bt, b=8)
    np.testing.assert_array_equal(np.concatenate([a["Z"], bb["Z"]], 2), full["Z"])
    np.testing.assert_array_equal(bb["W"], full["W"])


def test_update_rank_at_most_b():
    rng = np.random.default_rng(15)
    d, b = 16, 4
    Q, K, V, eta, W0, c0, g, bt = _rand_linear(rng, B=1, H=1, T=b, d=d)
    r = oracle.ttt_linear(Q, K, V, eta, W0, c0, g, bt, b=b)
    s = np.linalg.svd(r["W"][0, 0] - W0[0, 0], compute_uv=False)
    assert np.sum(s > 1e-10 * s[0]) <= b


def test_shared_w0_equals_broadcast():
    rng = np.random.default_rng(16)
    Q, K, V, eta, W0, c0, g, bt = _rand_linear(rng, B=3, shared=True)
    a = oracle.ttt_linear(Q, K, V, eta, W0, c0, g, bt, b=4)
    bb = oracle.ttt_linear(Q, K, V, eta, np.repeat(W0, 3, 0), np.repeat(c0, 3, 0), g, bt, b=4)
    for f in a:
        np.testing.assert_array_equal(a[f], bb[f])


def test_rejects_ragged_T():
    rng = np.random.default_rng(17)
    args = _rand_linear(rng, T=30)
    with pytest.raises(ValueError):
        oracle.ttt_linear(*args, b=4)


# ---------------------------------------------------------------- output rules
# The anchor rule (every prediction of mini-batch i made with W_{i-1}, the E2E
# review's section 2.3) and the key rule (the review's simplified output rule,
# Eq. 9: z_t = f(k_t; W_{i-1})) change only the output. Pins: the weight
# trajectory and inner loss are bit-identical under every rule; each output is
# the library LayerNorm / tanh-GELU forward at the anchor W_{i-1} (taken from
# the prefix-rule state after the first i batches, itself pinned above); under
# the key rule the output minus v is the inner residual, so loss == inner_loss.

def _anchor_states_linear(Q, K, V, eta, W0, c0, g, bt, b):
    """W_{i-1}, c_{i-1} for every batch i from prefix-rule runs over the first i batches."""
    T = Q.shape[2]
    out = []
    for i in range(T // b):
        if i == 0:
            out.append((np.broadcast_to(W0, (Q.shape[0],) + W0.shape[1:]),
                        np.broadcast_to(c0, (Q.shape[0],) + c0.shape[1:])))
        else:
            r = oracle.ttt_linear(Q[:, :, :i * b], K[:, :, :i * b], V[:, :, :i * b], eta[:, :, :i * b],
                                  W0, c0, g, bt, b=b)
            out.append((r["W"], r["c"]))
    return out


@pytest.mark.parametrize("rule", ["anchor", "key"])
@pytest.mark.parametrize("b", [1, 4])
def test_output_rule_is_library_forward_at_anchor_linear(rule, b):
    rng = np.random.default_rng(40 + b)
    Q, K, V, eta, W0, c0, g, bt = _rand_linear(rng, B=2, H=2, T=16, d=6)
    r = oracle.ttt_linear(Q, K, V, eta, W0, c0, g, bt, b=b, rule=rule)
    X = K if rule == "key" else Q
    for i, (Wa, ca) in enumerate(_anchor_states_linear(Q, K, V, eta, W0, c0, g, bt, b)):
        for bi in range(2):
            for hi in range(2):
                for t in range(i * b, (i + 1) * b):
                    z = _torch_f_linear(torch.tensor(Wa[bi, hi]), torch.tensor(ca[bi, hi]),
                                        torch.tensor(X[bi, hi, t]), torch.tensor(g[hi]), torch.tensor(bt[hi]),
                                        1e-6, True).numpy()
                    np.testing.assert_allclose(r["Z"][bi, hi, t], z, rtol=0, atol=1e-12)


@pytest.mark.parametrize("rule", ["anchor", "key"])
def test_output_rule_is_library_forward_at_anchor_mlp(rule):
    rng = np.random.default_rng(44)
    Q, K, V, eta, W1, c1, W2, c2, g, bt = _rand_mlp(rng, T=12)
    b = 4
    r = oracle.ttt_mlp(Q, K, V, eta, W1, c1, W2, c2, g, bt, b=b, rule=rule)
    X = K if rule == "key" else Q
    for i in range(3):
        if i == 0:
            st = dict(W1=W1, c1=c1, W2=W2, c2=c2)
        else:
            sl = slice(0, i * b)
            st = oracle.ttt_mlp(Q[:, :, sl], K[:, :, sl], V[:, :, sl], eta[:, :, sl], W1, c1, W2, c2, g, bt, b=b)
        for hi in range(2):
            for t in range(i * b, (i + 1) * b):
                z = _torch_f_mlp(*(torch.tensor(st[n][0, hi]) for n in ("W1", "c1", "W2", "c2")),
                                 torch.tensor(X[0, hi, t]), torch.tensor(g[hi]), torch.tensor(bt[hi]), 1e-6,
                                 True).numpy()
                np.testing.assert_allclose(r["Z"][0, hi, t], z, rtol=0, atol=1e-12)


@pytest.mark.parametrize("rule", ["anchor", "key"])
def test_output_rule_leaves_trajectory_unchanged(rule):
    rng = np.random.default_rng(46)
    Q, K, V, eta, W0, c0, g, bt = _rand_linear(rng, T=32, d=8)
    p = oracle.ttt_linear(Q, K, V, eta, W0, c0, g, bt, b=8)
    r = oracle.ttt_linear(Q, K, V, eta, W0, c0, g, bt, b=8, rule=rule)
    for f in ("W", "c", "inner_loss"):
        np.testing.assert_array_equal(r[f], p[f])
    assert np.abs(r["Z"] - p["Z"]).max() > 1e-3   # the outputs do differ
    args = _rand_mlp(rng, T=8)
    pm = oracle.ttt_mlp(*args, b=4)
    rm = oracle.ttt_mlp(*args, b=4, rule=rule)
    for f in ("W1", "c1", "W2", "c2", "inner_loss"):
        np.testing.assert_array_equal(rm[f], pm[f])


def test_key_rule_output_is_inner_prediction():
    rng = np.random.default_rng(47)
    Q, K, V, eta, W0, c0, g, bt = _rand_linear(rng, T=32, d=8)
    r = oracle.ttt_linear(None, K, V, eta, W0, c0, g, bt, b=8, rule="key")
    np.testing.assert_allclose(r["loss"], r["inner_loss"], rtol=1e-12, atol=0)
    rm = oracle.ttt_mlp(None, *(_rand_mlp(rng, T=8)[1:]), b=4, rule="key")
    np.testing.assert_allclose(rm["loss"], rm["inner_loss"], rtol=1e-12, atol=0)


@pytest.mark.parametrize("rule", ["anchor", "key"])
@pytest.mark.parametrize("b", [1, 4, 16])
def test_primal_equals_dual_output_rules(rule, b):
    rng = np.random.default_rng(48 + b)
    Q, K, V, eta, W0, c0, g, bt = _rand_linear(rng, T=32, d=8)
    p = oracle.ttt_linear(Q, K, V, eta, W0, c0, g, bt, b=b, rule=rule)
    dd = dual.ttt_linear_dual(Q, K, V, eta, W0, c0, g, bt, b=b, rule=rule)
    for f in p:
        np.testing.assert_allclose(dd[f], p[f], rtol=1e-11, atol=1e-11)
    args = _rand_mlp(rng, T=8)
    pm = oracle.ttt_mlp(*args, b=4, rule=rule)
    dm = dual.ttt_mlp_dual(*args, b=4, rule=rule)
    for f in pm:
        np.testing.assert_allclose(dm[f], pm[f], rtol=1e-11, atol=1e-11)


# ---------------------------------------------------------------- partial last mini-batch
# A final mini-batch of T % b < b tokens is emitted but not committed (the E2E
# review's section 2.3.2: a gradient step only once the decoded tokens fill a
# mini-batch). Pins: its outputs and losses equal the first rows of the same
# batch completed later (causality of every rule); the state equals the state
# of the committed prefix alone; committing later through the resume path gives
# the single-call result; with T < b the anchor output is the library forward at W_0.

@pytest.mark.parametrize("rule", ["prefix", "anchor", "key"])
@pytest.mark.parametrize("b,T", [(4, 14), (8, 5), (16, 37)])
def test_partial_tail_linear(rule, b, T):
    rng = np.random.default_rng(60 + b + T)
    Q, K, V, eta, W0, c0, g, bt = _rand_linear(rng, T=-(-T // b) * b, d=8)
    tc = (T // b) * b
    full = oracle.ttt_linear(Q, K, V, eta, W0, c0, g, bt, b=b, rule=rule)
    part = oracle.ttt_linear(Q[:, :, :T], K[:, :, :T], V[:, :, :T], eta[:, :, :T], W0, c0, g, bt, b=b, rule=rule,
                             partial_tail=True)
    for f in ("Z", "loss", "inner_loss"):
        np.testing.assert_array_equal(part[f], full[f][:, :, :T])
    if tc:
        pre = oracle.ttt_linear(Q[:, :, :tc], K[:, :, :tc], V[:, :, :tc], eta[:, :, :tc], W0, c0, g, bt, b=b,
                                rule=rule)
        np.testing.assert_array_equal(part["W"], pre["W"])
        np.testing.assert_array_equal(part["c"], pre["c"])
    else:
        np.testing.assert_array_equal(part["W"], np.broadcast_to(W0, part["W"].shape))
    # commit later: resume from the returned state with the completed batch
    rest = oracle.ttt_linear(Q[:, :, tc:], K[:, :, tc:], V[:, :, tc:], eta[:, :, tc:], part["W"], part["c"], g, bt,
                             b=b, rule=rule)
    np.testing.assert_array_equal(rest["W"], full["W"])
    np.testing.assert_array_equal(rest["Z"], full["Z"][:, :, tc:])
    d = dual.ttt_linear_dual(Q[:, :, :T], K[:, :, :T], V[:, :, :T], eta[:, :, :T], W0, c0, g, bt, b=b, rule=rule,
                             partial_tail=True)
    for f in part:
        np.testing.assert_allclose(d[f], part[f], rtol=1e-11, atol=1e-11)


def test_partial_only_batch_anchor_is_library_forward():
    rng = np.random.default_rng(70)
    Q, K, V, eta, W0, c0, g, bt = _rand_linear(rng, B=1, H=2, T=5, d=6)
    r = oracle.ttt_linear(Q, K, V, eta, W0, c0, g, bt, b=16, rule="anchor", partial_tail=True)
    for hi in range(2):
        for t in range(5):
            z = _torch_f_linear(torch.tensor(W0[0, hi]), torch.tensor(c0[0, hi]), torch.tensor(Q[0, hi, t]),
                                torch.tensor(g[hi]), torch.tensor(bt[hi]), 1e-6, True).numpy()
            np.testing.assert_allclose(r["Z"][0, hi, t], z, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(r["W"][0], W0[0])


@pytest.mark.parametrize("rule", ["prefix", "anchor"])
def test_partial_tail_mlp(rule):
    rng = np.random.default_rng(71)
    args = list(_rand_mlp(rng, T=12))
    b, T = 4, 10
    full = oracle.ttt_mlp(*args, b=b, rule=rule)
    cut = [a[:, :, :T] for a in args[:4]] + args[4:]
    part = oracle.ttt_mlp(*cut, b=b, rule=rule, partial_tail=True)
    for f in ("Z", "loss", "inner_loss"):
        np.testing.assert_array_equal(part[f], full[f][:, :, :T])
    pre = oracle.ttt_mlp(*([a[:, :, :8] for a in args[:4]] + args[4:]), b=b, rule=rule)
    for f in ("W1", "c1", "W2", "c2"):
        np.testing.assert_array_equal(part[f], pre[f])
    dm = dual.ttt_mlp_dual(*cut, b=b, rule=rule, partial_tail=True)
    for f in part:
        np.testing.assert_allclose(dm[f], part[f], rtol=1e-11, atol=1e-11)


# ---------------------------------------------------------------- learning-rate gate
# eta = eta_base * sigmoid(theta_lr . x) from the gate logits: pinned by its closed
# forms (logit 0 gives eta_base / 2; the gate saturates at eta_base; sigmoid(-z) =
# 1 - sigmoid(z)) and by the run it must reproduce: the gated oracle equals the
# oracle given those learning rates directly.

def test_gate_closed_forms():
    z = np.array([0.0, 40.0, -40.0, 1.3, -1.3])
    e = oracle.eta_from_gate(z, 0.7)
    assert e[0] == 0.35
    np.testing.assert_allclose(e[1], 0.7, rtol=1e-15)
    assert 0.0 < e[2] < 1e-17
    np.testing.assert_allclose(e[3] + e[4], 0.7, rtol=1e-15)


def test_gate_logit_zero_is_half_base():
    rng = np.random.default_rng(80)
    Q, K, V, eta, W0, c0, g, bt = _rand_linear(rng, T=16, d=6)
    a = oracle.ttt_linear(Q, K, V, np.zeros_like(eta), W0, c0, g, bt, b=4, eta_gate=True, eta_base=0.8)
    bb = oracle.ttt_linear(Q, K, V, np.full_like(eta, 0.4), W0, c0, g, bt, b=4)
    for f in a:
        np.testing.assert_array_equal(a[f], bb[f])
