"""fp64 CPU oracle of the test-time-training (TTT) inner loop.

TEST INFRASTRUCTURE. Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The CUDA library
(``test_weight_sequence_ttt_b300``) never imports it, and the two share no code.

Two independent implementations of the same method live here:

* ``ttt_linear`` / ``ttt_mlp`` -- the primal token loop in plain C
  (``ttt_oracle.c``), fp64, one chain per OpenMP thread. Steps follow the
  "TTT layer" section of the Test-Time Training survey page (Eq. 2 update,
  Eq. 4 loss, Eq. 5 output) with the mini-batch rule of Eq. 5 of the
  End-to-End Test-Time Training review (section 2.3).
* ``dual.ttt_linear_dual`` / ``dual.ttt_mlp_dual`` -- the mini-batch matrix
  ("dual") form in numpy, written separately; it never materialises the
  per-token gradients.

Both are pinned against things other than themselves in
``tests/test_oracle_pins.py`` (closed forms, autograd, finite differences,
Theorem 1 of the survey's "relation to attention" section, library LayerNorm
and GELU).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ttt_oracle.c")
_LIB = os.path.join(_HERE, "libttt_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile ``ttt_oracle.c`` into ``libttt_oracle.so`` (gcc, -O2, OpenMP).

    No fast-math: the oracle keeps IEEE double semantics."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.oracle_ttt_linear.restype = None
            lib.oracle_ttt_linear.argtypes = (
                [ctypes.c_int] * 8 + [_dp] * 6 + [ctypes.c_long] * 2 + [_dp] * 2
                + [ctypes.c_double] + [_dp] * 5 + [ctypes.c_int]
            )
            lib.oracle_ttt_mlp.restype = None
            lib.oracle_ttt_mlp.argtypes = (
                [ctypes.c_int] * 9 + [_dp] * 8 + [ctypes.c_long] * 3 + [_dp] * 2
                + [ctypes.c_double] + [_dp] * 7 + [ctypes.c_int]
            )
            lib.oracle_linear_token_grad.restype = ctypes.c_double
            lib.oracle_linear_token_grad.argtypes = (
                [ctypes.c_int] * 2 + [_dp] * 6 + [ctypes.c_double] + [_dp] * 2
            )
            lib.oracle_mlp_token_grad.restype = ctypes.c_double
            lib.oracle_mlp_token_grad.argtypes = (
                [ctypes.c_int] * 3 + [_dp] * 8 + [ctypes.c_double] + [_dp] * 4
            )
            lib.oracle_max_threads.restype = ctypes.c_int
            lib.oracle_max_threads.argtypes = []
            _lib = lib
    return _lib


def max_threads() -> int:
    return _load().oracle_max_threads()


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a):
    return a.ctypes.data_as(_dp)


RULES = {"prefix": 0, "anchor": 1, "key": 2}


def eta_from_gate(logit, eta_base):
    """The learnable learning-rate gate of the survey's "TTT layer" section,
    eta = eta_base * sigmoid(theta_lr . x), from the gate logits theta_lr . x (fp64)."""
    z = np.asarray(logit, np.float64)
    return float(eta_base) / (1.0 + np.exp(-z))


def _rule(rule):
    if rule not in RULES:
        raise ValueError("rule must be one of %s" % sorted(RULES))
    return RULES[rule]


def _init_stride(a, B, per):
    """Batch stride (elements) of an initial-weight array [B or 1, H, ...]."""
    if a.shape[0] == 1 and B != 1:
        return 0
    assert a.shape[0] == B, "initial weights need a leading dim of B or 1"
    return per


def ttt_linear(Q, K, V, eta, W0, c0, ln_g, ln_b, *, b, eps=1e-6, ln_res=True, nthreads=0, rule="prefix",
               partial_tail=False, eta_gate=False, eta_base=1.0):
    """TTT-Linear primal token loop in fp64.

    Q, K, V [B,H,T,d]; eta [B,H,T]; W0 [B|1,H,d,d] (f_res(x) = W x + c);
    c0 [B|1,H,d]; ln_g, ln_b [H,d]. T must be a multiple of b.
    Returns a dict with Z [B,H,T,d], W, c (final state), loss (L_t =
    ||z_t - v_t||^2) and inner_loss (l_t at the mini-batch anchor W_{i-1}).
    ``rule``: "prefix" z_t = f(q_t; W_t), "anchor" f(q_t; W_{i-1}), "key"
    f(k_t; W_{i-1}) (Q is then not read and may be None). With ``partial_tail``
    T need not be a multiple of b: the last T % b tokens are emitted but not
    committed (the final state is the one after the last full mini-batch).
    With ``eta_gate``, ``eta`` holds the gate logits and the learning rates are
    eta_base * sigmoid(logit)."""
    if Q is None:
        Q = K
    if eta_gate:
        eta = eta_from_gate(eta, eta_base)
    Q, K, V, eta, W0, c0, ln_g, ln_b = map(_f64, (Q, K, V, eta, W0, c0, ln_g, ln_b))
    B, H, T, d = Q.shape
    if T % b and not partial_tail:
        raise ValueError("T must be a multiple of the mini-batch size b")
    Z = np.empty_like(Q)
    W = np.empty((B, H, d, d))
    c = np.empty((B, H, d))
    loss = np.empty((B, H, T))
    inner = np.empty((B, H, T))
    _load().oracle_ttt_linear(
        B, H, T, d, b, int(bool(ln_res)), _rule(rule), int(bool(partial_tail)), _p(Q), _p(K), _p(V), _p(eta),
        _p(W0), _p(c0),
        _init_stride(W0, B, H * d * d), _init_stride(c0, B, H * d), _p(ln_g), _p(ln_b),
        float(eps), _p(Z), _p(W), _p(c), _p(loss), _p(inner), int(nthreads),
    )
    return dict(Z=Z, W=W, c=c, loss=loss, inner_loss=inner)


def ttt_mlp(Q, K, V, eta, W1, c1, W2, c2, ln_g, ln_b, *, b, eps=1e-6, ln_res=True, nthreads=0,
            rule="prefix", partial_tail=False, eta_gate=False, eta_base=1.0):
    """TTT-MLP primal token loop in fp64; f_res(x) = W2 gelu_tanh(W1 x + c1) + c2.

    W1 [B|1,H,h,d], c1 [B|1,H,h], W2 [B|1,H,d,h], c2 [B|1,H,d]; ``rule`` as
    for ``ttt_linear`` (so are ``partial_tail``, ``eta_gate`` and ``eta_base``)."""
    if Q is None:
        Q = K
    if eta_gate:
        eta = eta_from_gate(eta, eta_base)
    Q, K, V, eta, W1, c1, W2, c2, ln_g, ln_b = map(_f64, (Q, K, V, eta, W1, c1, W2, c2, ln_g, ln_b))
    B, H, T, d = Q.shape
    h = W1.shape[-2]
    if T % b and not partial_tail:
        raise ValueError("T must be a multiple of the mini-batch size b")
    if W1.shape[0] != W2.shape[0]:
        raise ValueError("W1 and W2 must share their leading dim")
    Z = np.empty_like(Q)
    W1o = np.empty((B, H, h, d))
    W2o = np.empty((B, H, d, h))
    c1o = np.empty((B, H, h))
    c2o = np.empty((B, H, d))
    loss = np.empty((B, H, T))
    inner = np.empty((B, H, T))
    _load().oracle_ttt_mlp(
        B, H, T, d, h, b, int(bool(ln_res)), _rule(rule), int(bool(partial_tail)), _p(Q), _p(K), _p(V), _p(eta),
        _p(W1), _p(c1),
        _p(W2), _p(c2), _init_stride(W1, B, H * h * d), _init_stride(c1, B, H * h),
        _init_stride(c2, B, H * d), _p(ln_g), _p(ln_b), float(eps), _p(Z), _p(W1o), _p(c1o),
        _p(W2o), _p(c2o), _p(loss), _p(inner), int(nthreads),
    )
    return dict(Z=Z, W1=W1o, c1=c1o, W2=W2o, c2=c2o, loss=loss, inner_loss=inner)


def linear_token_grad(W, c, k, v, ln_g, ln_b, *, eps=1e-6, ln_res=True):
    """Loss of Eq. 4 for one token and its gradient (dW, dc) at (W, c)."""
    W, c, k, v, ln_g, ln_b = map(_f64, (W, c, k, v, ln_g, ln_b))
    d = k.shape[0]
    dW = np.empty((d, d))
    dc = np.empty(d)
    l = _load().oracle_linear_token_grad(
        d, int(bool(ln_res)), _p(W), _p(c), _p(k), _p(v), _p(ln_g), _p(ln_b), float(eps), _p(dW), _p(dc)
    )
    return l, dW, dc


def mlp_token_grad(W1, c1, W2, c2, k, v, ln_g, ln_b, *, eps=1e-6, ln_res=True):
    """Loss of Eq. 4 for one token through the MLP and its gradient."""
    W1, c1, W2, c2, k, v, ln_g, ln_b = map(_f64, (W1, c1, W2, c2, k, v, ln_g, ln_b))
    h, d = W1.shape
    dW1 = np.empty((h, d))
    dc1 = np.empty(h)
    dW2 = np.empty((d, h))
    dc2 = np.empty(d)
    l = _load().oracle_mlp_token_grad(
        d, h, int(bool(ln_res)), _p(W1), _p(c1), _p(W2), _p(c2), _p(k), _p(v), _p(ln_g),
        _p(ln_b), float(eps), _p(dW1), _p(dc1), _p(dW2), _p(dc2)
    )
    return l, dW1, dc1, dW2, dc2
