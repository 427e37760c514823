"""Partial last mini-batch (decode / chunked prefill), GPU.

With partial_tail the last T % b tokens are emitted (Z, loss, inner_loss) but
not committed (the E2E review's section 2.3.2). On every kernel family:
the outputs follow the fp64 oracle within the path's tolerance; the final
state is bit-identical to a call on the committed prefix alone; and, because
outputs are causal, the tail's outputs are bit-identical to the first rows the
completed mini-batch gives later.
"""
import pytest
import torch

import test_weight_sequence_ttt_b300 as ttt
from test_weight_sequence_ttt_b300.inputs import WORKLOADS, make_inputs

from _util import TOL, compare, dev, oracle_linear, oracle_mlp, rel_err, to_np

pytestmark = pytest.mark.gpu

# (d, b, T, io, kind): split d=64 (b=16, b=4), merged d=128 (b=16, b=8), the
# b=64 / b=32 paths (tail of several super-steps; tail only), fp32 kernels.
LIN = [(64, 16, 37, "bf16", 2), (64, 4, 42, "bf16", 2), (64, 16, 9, "bf16", 2), (128, 16, 23, "bf16", 2),
       (64, 16, 1, "bf16", 2), (64, 16, 47, "bf16", 2),
       (128, 8, 45, "bf16", 2), (64, 64, 100, "bf16", 2), (128, 32, 40, "bf16", 2), (64, 64, 20, "bf16", 2),
       (64, 256, 600, "bf16", 2), (128, 128, 300, "bf16", 2),
       (16, 16, 21, "f32", 1), (32, 16, 40, "bf16", 1)]


def _run_lin(inp, T, rule="prefix", tail=True):
    d = dev(inp)
    sl = lambda x: x[:, :, :T].contiguous()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = ttt.ttt_linear_forward(sl(d["Q"]), sl(d["K"]), sl(d["V"]), sl(d["eta"]), d["W0"], d["c0"], d["ln_g"],
                               d["ln_b"], mb=inp["b"], eps=inp["eps"], status=st, out_rule=rule, partial_tail=tail)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return o


@pytest.mark.parametrize("rule", ["prefix", "anchor"])
@pytest.mark.parametrize("d,b,T,io,kind", LIN)
def test_linear_partial_tail(rule, d, b, T, io, kind, linear_form):
    assert ttt.linear_kernel_kind(ttt.BF16 if io == "bf16" else ttt.F32, d, b) == kind
    Tfull = -(-T // b) * b
    w = WORKLOADS["linear_b8h12_d64_t2k"].with_(B=2, H=2, T=Tfull, d=d, b=b, io=io, seed=300 + T)
    inp = make_inputs(w)
    got = _run_lin(inp, T, rule)
    cut = dict(inp)
    for k in ("Q", "K", "V", "eta"):
        cut[k] = inp[k][:, :, :T]
    import oracle
    ref = oracle.ttt_linear(*(to_np(cut[k]) for k in ("Q", "K", "V", "eta", "W0", "c0", "ln_g", "ln_b")),
                            b=b, eps=inp["eps"], rule=rule, partial_tail=True)
    compare(got, ref, ("Z", "W", "c", "loss", "inner_loss"), TOL[io])
    tc = (T // b) * b
    if tc:   # the state is the committed prefix's, bit for bit
        pre = _run_lin(inp, tc, rule, tail=False)
        assert torch.equal(got["W"], pre["W"]) and torch.equal(got["c"], pre["c"])
    if rule == "prefix":   # the tail's outputs are the completed batch's first rows
        full = _run_lin(inp, Tfull, rule, tail=False)
        for k in ("Z", "loss", "inner_loss"):
            assert torch.equal(got[k], full[k][:, :, :T]), k


@pytest.mark.parametrize("d,h,b,T,io", [(64, 256, 16, 40, "bf16"), (64, 256, 16, 7, "bf16"), (64, 256, 16, 1, "bf16"),
                                        (64, 256, 16, 17, "bf16"), (64, 256, 16, 63, "bf16"), (16, 48, 4, 10, "f32")])
def test_mlp_partial_tail(d, h, b, T, io, mlp_form):
    Tfull = -(-T // b) * b
    w = WORKLOADS["mlp_b4h12_d64_t8k"].with_(B=2, H=2, T=Tfull, d=d, hidden=h, b=b, io=io, seed=400 + T)
    inp = make_inputs(w)
    dd = dev(inp)

    def run(TT, tail):
        sl = lambda x: x[:, :, :TT].contiguous()
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        o = ttt.ttt_mlp_forward(sl(dd["Q"]), sl(dd["K"]), sl(dd["V"]), sl(dd["eta"]), dd["W1"], dd["c1"], dd["W2"],
                                dd["c2"], dd["ln_g"], dd["ln_b"], mb=b, eps=inp["eps"], status=st, partial_tail=tail)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        return o

    got = run(T, True)
    import oracle
    cut = [to_np(inp[k][:, :, :T]) for k in ("Q", "K", "V", "eta")]
    ref = oracle.ttt_mlp(*cut, *(to_np(inp[k]) for k in ("W1", "c1", "W2", "c2", "ln_g", "ln_b")), b=b,
                         eps=inp["eps"], partial_tail=True)
    compare(got, ref, ("Z", "W1", "c1", "W2", "c2", "loss", "inner_loss"), TOL[io])
    tc = (T // b) * b
    if tc:
        pre = run(tc, False)
        for k in ("W1", "c1", "W2", "c2"):
            assert torch.equal(got[k], pre[k]), k
    full = run(Tfull, False)
    for k in ("Z", "loss", "inner_loss"):
        assert torch.equal(got[k], full[k][:, :, :T]), k


@pytest.mark.parametrize("name", ["linear_b8h12_d64_decode15", "mlp_b4h12_d64_decode15"])
def test_decode_workload_full_size(name):
    """The decode-step workloads at their bench size, every chain against the oracle."""
    w = WORKLOADS[name]
    inp = make_inputs(w)
    d = dev(inp)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    if w.variant == "linear":
        got = ttt.ttt_linear_forward(d["Q"], d["K"], d["V"], d["eta"], d["W0"], d["c0"], d["ln_g"], d["ln_b"],
                                     mb=w.b, eps=w.eps, status=st, partial_tail=True)
        ref = oracle_linear(inp, partial_tail=True)
        keys = ("Z", "W", "c", "loss", "inner_loss")
    else:
        got = ttt.ttt_mlp_forward(d["Q"], d["K"], d["V"], d["eta"], d["W1"], d["c1"], d["W2"], d["c2"], d["ln_g"],
                                  d["ln_b"], mb=w.b, eps=w.eps, status=st, partial_tail=True)
        ref = oracle_mlp(inp, partial_tail=True)
        keys = ("Z", "W1", "c1", "W2", "c2", "loss", "inner_loss")
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    compare(got, ref, keys, TOL["bf16"])
