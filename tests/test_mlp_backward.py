"""GPU parity of the TTT-MLP backward (``ttt_mlp_backward``) against the fp64
backward oracle (``oracle.backward.ttt_mlp_backward``, pinned by finite
differences).

Each gradient tensor is compared element by element: max |err| <= TOL_BWD * RMS
of the oracle's tensor, the bound of the TTT-Linear backward (fp32 arithmetic
throughout). The full-length chain (T = 8192: 512 mini-batches whose adjoints
the reverse sweep accumulates one after the other through the two layers and
the GELU's second derivative) is held to TOL_BWD_FULL instead: there the fp32
rounding of the long reverse accumulation reaches about 3e-4 on dK, dV and
deta (measured), while every shorter case stays under 1e-4. Sizes span several mini-batches, b in {1, 4, 16}, widths that are
not multiples of the warp, bf16 inputs, the learning-rate gate, optional seeds
and per-sequence initial weights; the benchmark's TTT-MLP workload runs on the
GPU with one sampled chain checked against the oracle at full length. b = 16
runs the two-CTA cluster kernel where h is a multiple of 8 and the single-CTA
kernel otherwise; both are covered.
"""
import numpy as np
import pytest
import torch

import test_weight_sequence_ttt_b300 as ttt
from oracle.backward import ttt_mlp_backward as oracle_bwd
from test_weight_sequence_ttt_b300.inputs import WORKLOADS, make_cotangents, make_inputs

from _util import rel_err, to_np

pytestmark = pytest.mark.gpu

TOL_BWD = 1e-4
TOL_BWD_FULL = 1e-3
KEYS = ["dQ", "dK", "dV", "deta", "dW1", "dc1", "dW2", "dc2", "dln_g", "dln_b"]
INS = ["Q", "K", "V", "eta", "W1", "c1", "W2", "c2", "ln_g", "ln_b"]
SEEDS = ["dW1_n", "dc1_n", "dW2_n", "dc2_n"]


def _case(B, H, T, d, h, b, io="f32", seed=0, gate=False, per_seq=False):
    rng = np.random.default_rng(seed)
    dt = torch.float32 if io == "f32" else torch.bfloat16

    def t(a, dtype=torch.float32):
        return torch.tensor(np.asarray(a), dtype=torch.float64).to(dtype)

    lead = B if per_seq else 1
    return dict(
        Q=t(rng.standard_normal((B, H, T, d)), dt), K=t(rng.standard_normal((B, H, T, d)), dt),
        V=t(rng.standard_normal((B, H, T, d)), dt),
        eta=t(rng.standard_normal((B, H, T)) if gate else rng.uniform(0.1, 1.0, (B, H, T))),
        W1=t(rng.standard_normal((lead, H, h, d)) * 0.6 / np.sqrt(d)), c1=t(rng.standard_normal((lead, H, h)) * 0.1),
        W2=t(rng.standard_normal((lead, H, d, h)) * 0.6 / np.sqrt(h)), c2=t(rng.standard_normal((lead, H, d)) * 0.1),
        ln_g=t(rng.uniform(0.5, 1.5, (H, d))), ln_b=t(rng.standard_normal((H, d)) * 0.1),
        dZ=t(rng.standard_normal((B, H, T, d)), dt),
        dW1_n=t(rng.standard_normal((B, H, h, d)) * 0.1), dc1_n=t(rng.standard_normal((B, H, h)) * 0.1),
        dW2_n=t(rng.standard_normal((B, H, d, h)) * 0.1), dc2_n=t(rng.standard_normal((B, H, d)) * 0.1),
        b=b, eps=1e-6,
    )


def _run(x, *, gate=False, eta_base=1.0, seeds=True, status=None):
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    kw = {k: (g[k] if seeds else None) for k in SEEDS}
    out = ttt.ttt_mlp_backward(*(g[k] for k in INS), g["dZ"], mb=x["b"], eps=x["eps"], eta_gate=gate,
                               eta_base=eta_base, status=status, **kw)
    torch.cuda.synchronize()
    return out


def _oracle(x, *, gate=False, eta_base=1.0, seeds=True):
    return oracle_bwd(*(to_np(x[k]) for k in INS), to_np(x["dZ"]),
                      *((to_np(x[k]) if seeds else None) for k in SEEDS), b=x["b"], eps=x["eps"],
                      eta_gate=gate, eta_base=eta_base)


def _compare(got, ref, sel=None, tol=TOL_BWD):
    errs = {}
    for k in KEYS:
        g = to_np(got[k])
        if sel is not None:
            g = g[sel]
        errs[k] = rel_err(g.reshape(ref[k].shape), ref[k])
    print(errs)
    bad = {k: e for k, e in errs.items() if not e <= tol}
    assert not bad, "max|err|/RMS above %.0e: %s (all: %s)" % (tol, bad, errs)
    return errs


@pytest.mark.parametrize("B,H,T,d,h,b,io", [
    (1, 2, 64, 16, 64, 16, "f32"), (1, 2, 64, 64, 256, 16, "f32"), (2, 1, 24, 8, 36, 4, "f32"),
    (1, 1, 12, 12, 20, 1, "f32"), (1, 2, 64, 64, 256, 16, "bf16"), (1, 1, 32, 40, 160, 8, "f32"),
    (1, 2, 48, 12, 20, 16, "f32"),   # b = 16 with h not a multiple of 8: the single-CTA kernel
])
def test_mlp_backward_matches_oracle(B, H, T, d, h, b, io):
    x = _case(B, H, T, d, h, b, io, seed=B * 100 + T + d + h + b)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _run(x, status=st)
    assert int(st.item()) == 0
    _compare(got, _oracle(x))


# d = 64, h = 256 runs the cluster kernel compiled for that shape; the others the runtime-sized one
@pytest.mark.parametrize("d,h", [(16, 64), (64, 256)])
def test_mlp_backward_gate_no_seeds_per_sequence(d, h):
    x = _case(2, 1, 32, d, h, 16, seed=31, gate=True, per_seq=True)
    _compare(_run(x, gate=True, eta_base=0.6, seeds=False), _oracle(x, gate=True, eta_base=0.6, seeds=False))


@pytest.mark.parametrize("d,h", [(32, 128), (64, 256)])
def test_mlp_backward_deterministic(d, h):
    x = _case(1, 2, 32, d, h, 16, seed=32)
    a, b_ = _run(x), _run(x)
    for k in KEYS:
        assert torch.equal(a[k], b_[k]), k


def test_mlp_backward_full_workload_sampled_chain():
    """The benchmark's TTT-MLP workload (bf16 Q/K/V, B=4, H=12, d=64, h=256,
    T=8192, b=16) on every chain; the oracle recomputes the last chain."""
    w = WORKLOADS["mlp_b4h12_d64_t8k"]
    x = dict(make_inputs(w), **make_cotangents(w))
    got = _run(x)
    ch = w.chains - 1
    si = make_inputs(w, chains=[ch])
    sc = make_cotangents(w, chains=[ch])
    ref = oracle_bwd(*(to_np(si[k]) for k in INS), to_np(sc["dZ"]), *(to_np(sc[k]) for k in SEEDS), b=w.b,
                     eps=w.eps)
    bi, hi = divmod(ch, w.H)
    _compare(got, ref, sel=(slice(bi, bi + 1), slice(hi, hi + 1)), tol=TOL_BWD_FULL)
