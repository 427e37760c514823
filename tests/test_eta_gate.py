"""Learning-rate gate in the kernels (GPU): with eta_gate the eta input holds
the gate logits theta_lr . x and every kernel family applies
eta = eta_base * sigmoid(logit) itself (tokens past T of a partial tail keep
eta = 0). Checked against the fp64 oracle with the same gate, and against the
kernel run given the learning rates that the input generator also returns.
"""
import pytest
import torch

import test_weight_sequence_ttt_b300 as ttt
from test_weight_sequence_ttt_b300.inputs import WORKLOADS, make_inputs

from _util import TOL, compare, dev, rel_err, to_np

pytestmark = pytest.mark.gpu
import oracle  # noqa: E402

LIN = [(64, 16, 48, "bf16"), (64, 4, 40, "bf16"), (128, 16, 48, "bf16"), (64, 64, 192, "bf16"), (64, 256, 512, "bf16"),
       (16, 16, 64, "f32"), (64, 16, 37, "bf16")]   # the last one with a partial tail


@pytest.mark.parametrize("d,b,T,io", LIN)
def test_linear_gate(d, b, T, io, linear_form):
    tail = T % b != 0
    w = WORKLOADS["linear_b8h12_d64_t2k"].with_(B=2, H=2, T=T, d=d, b=b, io=io, seed=600 + T, eta_base=0.8,
                                                partial_tail=tail)
    inp = make_inputs(w)
    dd = dev(inp)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = ttt.ttt_linear_forward(dd["Q"], dd["K"], dd["V"], dd["eta_logit"], dd["W0"], dd["c0"], dd["ln_g"],
                                 dd["ln_b"], mb=b, eps=w.eps, status=st, eta_gate=True, eta_base=0.8,
                                 partial_tail=tail)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = oracle.ttt_linear(*(to_np(inp[k]) for k in ("Q", "K", "V", "eta_logit", "W0", "c0", "ln_g", "ln_b")),
                            b=b, eps=w.eps, eta_gate=True, eta_base=0.8, partial_tail=tail)
    compare(got, ref, ("Z", "W", "c", "loss", "inner_loss"), TOL[io])
    # the same run given the learning rates directly agrees to fp32 rounding of the gate
    plain = ttt.ttt_linear_forward(dd["Q"], dd["K"], dd["V"], dd["eta"], dd["W0"], dd["c0"], dd["ln_g"],
                                   dd["ln_b"], mb=b, eps=w.eps, partial_tail=tail)
    torch.cuda.synchronize()
    assert rel_err(to_np(got["Z"]), to_np(plain["Z"])) <= 1e-3


@pytest.mark.parametrize("d,h,b,T,io", [(64, 256, 16, 48, "bf16"), (64, 256, 16, 40, "bf16"), (16, 48, 4, 24, "f32")])
def test_mlp_gate(d, h, b, T, io, mlp_form):
    tail = T % b != 0
    w = WORKLOADS["mlp_b4h12_d64_t8k"].with_(B=1, H=2, T=T, d=d, hidden=h, b=b, io=io, seed=700 + T, eta_base=0.6,
                                             partial_tail=tail)
    inp = make_inputs(w)
    dd = dev(inp)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = ttt.ttt_mlp_forward(dd["Q"], dd["K"], dd["V"], dd["eta_logit"], dd["W1"], dd["c1"], dd["W2"], dd["c2"],
                              dd["ln_g"], dd["ln_b"], mb=b, eps=w.eps, status=st, eta_gate=True, eta_base=0.6,
                              partial_tail=tail)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = oracle.ttt_mlp(*(to_np(inp[k]) for k in ("Q", "K", "V", "eta_logit", "W1", "c1", "W2", "c2", "ln_g",
                                                   "ln_b")), b=b, eps=w.eps, eta_gate=True, eta_base=0.6,
                         partial_tail=tail)
    compare(got, ref, ("Z", "W1", "c1", "W2", "c2", "loss", "inner_loss"), TOL[io])
