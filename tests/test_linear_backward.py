"""GPU parity of the TTT-Linear backward (``ttt_linear_backward``) against the
fp64 backward oracle (``oracle.backward``, pinned by finite differences).

Each gradient tensor is compared element by element: max |err| <= TOL_BWD * RMS
of the oracle's tensor, the fp32 forward path's bound. The default arithmetic
is fp32-grade: fp32 FFMA, or for d = 64, b = 16 tensor-core products in split
precision (three tf32 products per product, fp32 accumulation). math="tf32"
(one tf32 product each in the reverse sweep) is gated at TOL_TF32.

Sizes span several mini-batches, a head dim that is not a multiple of the warp
(d = 40), a mini-batch size that is not a power of two (b = 12), b = 1 and
b = 64, d = 128, bf16 inputs, the learning-rate gate, optional seeds and
per-sequence initial weights; the full workload of the benchmark runs on the GPU
with sampled chains checked against the oracle.
"""
import numpy as np
import pytest
import torch

import test_weight_sequence_ttt_b300 as ttt
from oracle.backward import ttt_linear_backward as oracle_bwd
from test_weight_sequence_ttt_b300.inputs import WORKLOADS, make_cotangents, make_inputs

from _util import rel_err, to_np

pytestmark = pytest.mark.gpu

TOL_BWD = 1e-4
# math="tf32" (d = 64, b = 16): reverse-sweep operands rounded to 10 mantissa bits
# (2^-11 relative each), accumulated in fp32 over every mini-batch of the reverse
# sweep: measured up to 1.5e-2 at T = 2048, gated at the bf16-operand bound
TOL_TF32 = 2e-2
KEYS = ["dQ", "dK", "dV", "deta", "dW0", "dc0", "dln_g", "dln_b"]


def _case(B, H, T, d, b, io="f32", seed=0, gate=False, per_seq=False):
    """Inputs with non-trivial LayerNorm, bias and initial weights (torch CPU)."""
    rng = np.random.default_rng(seed)
    dt = torch.float32 if io == "f32" else torch.bfloat16

    def t(a, dtype=torch.float32):
        return torch.tensor(np.asarray(a), dtype=torch.float64).to(dtype)

    lead = B if per_seq else 1
    return dict(
        Q=t(rng.standard_normal((B, H, T, d)), dt), K=t(rng.standard_normal((B, H, T, d)), dt),
        V=t(rng.standard_normal((B, H, T, d)), dt),
        eta=t(rng.standard_normal((B, H, T)) if gate else rng.uniform(0.1, 1.0, (B, H, T))),
        W0=t(rng.standard_normal((lead, H, d, d)) * 0.5 / np.sqrt(d)),
        c0=t(rng.standard_normal((lead, H, d)) * 0.1),
        ln_g=t(rng.uniform(0.5, 1.5, (H, d))), ln_b=t(rng.standard_normal((H, d)) * 0.1),
        dZ=t(rng.standard_normal((B, H, T, d)), dt), dW_n=t(rng.standard_normal((B, H, d, d)) * 0.1),
        dc_n=t(rng.standard_normal((B, H, d)) * 0.1), b=b, eps=1e-6,
    )


def _run(x, *, gate=False, eta_base=1.0, seeds=True, status=None, math="fp32"):
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    out = ttt.ttt_linear_backward(g["Q"], g["K"], g["V"], g["eta"], g["W0"], g["c0"], g["ln_g"], g["ln_b"],
                                  g["dZ"], mb=x["b"], dW_n=g["dW_n"] if seeds else None,
                                  dc_n=g["dc_n"] if seeds else None, eps=x["eps"], eta_gate=gate,
                                  eta_base=eta_base, status=status, math=math)
    torch.cuda.synchronize()
    return out


def _oracle(x, *, gate=False, eta_base=1.0, seeds=True):
    return oracle_bwd(*(to_np(x[k]) for k in ("Q", "K", "V", "eta", "W0", "c0", "ln_g", "ln_b", "dZ")),
                      to_np(x["dW_n"]) if seeds else None, to_np(x["dc_n"]) if seeds else None, b=x["b"],
                      eps=x["eps"], eta_gate=gate, eta_base=eta_base)


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


@pytest.mark.parametrize("B,H,T,d,b,io", [
    (2, 2, 64, 16, 16, "f32"), (1, 3, 128, 64, 16, "f32"), (1, 2, 96, 40, 12, "f32"),
    (2, 2, 48, 64, 1, "f32"), (1, 2, 256, 64, 32, "f32"), (1, 2, 256, 32, 64, "f32"),
    (1, 2, 64, 128, 16, "f32"), (1, 2, 256, 128, 16, "bf16"),
    (2, 2, 128, 64, 16, "bf16"), (1, 1, 16, 8, 16, "f32"),
    (1, 1, 32, 128, 8, "f32"),       # d = 128 on the general kernel
])
def test_backward_matches_oracle(B, H, T, d, b, io):
    x = _case(B, H, T, d, b, io, seed=B * 1000 + T + d + b)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _run(x, status=st)
    assert int(st.item()) == 0
    _compare(got, _oracle(x))


def test_backward_learning_rate_gate():
    x = _case(1, 2, 64, 64, 16, seed=7, gate=True)
    _compare(_run(x, gate=True, eta_base=0.7), _oracle(x, gate=True, eta_base=0.7))


def test_backward_without_state_seeds():
    x = _case(2, 1, 64, 32, 8, seed=8)
    _compare(_run(x, seeds=False), _oracle(x, seeds=False))


def test_backward_per_sequence_initial_weights():
    x = _case(2, 2, 64, 32, 16, seed=9, per_seq=True)
    _compare(_run(x), _oracle(x))


def test_backward_deterministic_and_chain_independent():
    x = _case(2, 3, 64, 64, 16, seed=10)
    a = _run(x)
    b_ = _run(x)
    for k in KEYS:
        assert torch.equal(a[k], b_[k]), k
    # chain (1, 2) alone gives the same bits as inside the batch
    one = {k: (v[1:2, 2:3].contiguous() if isinstance(v, torch.Tensor) and v.dim() >= 3 and v.shape[0] == 2
               else v) for k, v in x.items()}
    one["W0"] = x["W0"][:, 2:3].contiguous()
    one["c0"] = x["c0"][:, 2:3].contiguous()
    one["ln_g"] = x["ln_g"][2:3].contiguous()
    one["ln_b"] = x["ln_b"][2:3].contiguous()
    c = _run(one)
    for k in KEYS:
        assert torch.equal(c[k][0, 0], a[k][1, 2]), k


def test_backward_full_workload_sampled_chains():
    """The benchmark's TTT-Linear workload (bf16 Q/K/V, B=8, H=12, d=64, T=2048,
    b=16) on every chain; the oracle recomputes two sampled chains."""
    w = WORKLOADS["linear_b8h12_d64_t2k"]
    inp = make_inputs(w)
    cot = make_cotangents(w)
    x = dict(inp, **cot)
    got = _run(x)
    for ch in (5, w.chains - 1):
        si = make_inputs(w, chains=[ch])
        sc = make_cotangents(w, chains=[ch])
        ref = oracle_bwd(*(to_np(si[k]) for k in ("Q", "K", "V", "eta", "W0", "c0", "ln_g", "ln_b")),
                         to_np(sc["dZ"]), to_np(sc["dW_n"]), to_np(sc["dc_n"]), b=w.b, eps=w.eps)
        bi, hi = divmod(ch, w.H)
        _compare(got, ref, sel=(slice(bi, bi + 1), slice(hi, hi + 1)))


def test_backward_reports_nonfinite_gradients():
    x = _case(1, 1, 32, 16, 16, seed=11)
    x["dW_n"][0, 0, 0, 0] = float("inf")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    _run(x, status=st)
    assert int(st.item()) == 8  # TTT_ERR_NONFINITE


def test_backward_host_pointer_rejected():
    x = _case(1, 1, 32, 16, 16, seed=12)
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    ws = torch.empty(ttt.linear_backward_workspace_bytes(1, 1, 32, 16, 16), dtype=torch.uint8)  # host memory
    with pytest.raises(ValueError):
        ttt.ttt_linear_backward(g["Q"], g["K"], g["V"], g["eta"], g["W0"], g["c0"], g["ln_g"], g["ln_b"],
                                g["dZ"], mb=16, workspace=ws)


# ---------------------------------------------------------------- tf32 tensor-core kernel (d = 64, b = 16)

@pytest.mark.parametrize("B,H,T,d,io", [(1, 3, 128, 64, "f32"), (2, 2, 128, 64, "bf16"), (1, 1, 16, 64, "f32"),
                                         (2, 1, 512, 64, "bf16"), (1, 2, 256, 128, "bf16"), (1, 1, 64, 128, "f32")])
def test_backward_tf32_matches_oracle(B, H, T, d, io):
    x = _case(B, H, T, d, 16, io, seed=B * 1000 + T + 2 + d)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _run(x, status=st, math="tf32")
    assert int(st.item()) == 0
    _compare(got, _oracle(x), tol=TOL_TF32)


def test_backward_tf32_gate_no_seeds_per_sequence():
    x = _case(2, 2, 64, 64, 16, seed=13, gate=True, per_seq=True)
    _compare(_run(x, gate=True, eta_base=0.7, seeds=False, math="tf32"),
             _oracle(x, gate=True, eta_base=0.7, seeds=False), tol=TOL_TF32)


def test_backward_tf32_deterministic_and_other_sizes_fall_back():
    x = _case(2, 3, 64, 64, 16, seed=14)
    a, b_ = _run(x, math="tf32"), _run(x, math="tf32")
    for k in KEYS:
        assert torch.equal(a[k], b_[k]), k
    # sizes without a tensor-core kernel run the fp32 one: identical results
    y = _case(1, 2, 64, 32, 16, seed=15)
    f, t = _run(y), _run(y, math="tf32")
    for k in KEYS:
        assert torch.equal(f[k], t[k]), k


def test_backward_tf32_full_workload_sampled_chains():
    """The benchmark's TTT-Linear workload on the tf32 kernel, two sampled chains."""
    w = WORKLOADS["linear_b8h12_d64_t2k"]
    x = dict(make_inputs(w), **make_cotangents(w))
    got = _run(x, math="tf32")
    for ch in (5, w.chains - 1):
        si = make_inputs(w, chains=[ch])
        sc = make_cotangents(w, chains=[ch])
        ref = oracle_bwd(*(to_np(si[k]) for k in ("Q", "K", "V", "eta", "W0", "c0", "ln_g", "ln_b")),
                         to_np(sc["dZ"]), to_np(sc["dW_n"]), to_np(sc["dc_n"]), b=w.b, eps=w.eps)
        bi, hi = divmod(ch, w.H)
        _compare(got, ref, sel=(slice(bi, bi + 1), slice(hi, hi + 1)), tol=TOL_TF32)
