"""Output-rule variants (GPU): the anchor rule z_t = f(q_t; W_{i-1}) of the
End-to-End TTT review's section 2.3 and its simplified output rule, Eq. 9,
z_t = f(k_t; W_{i-1}), against the fp64 oracle, on every kernel family.

The weight trajectory does not depend on the output rule, so on the GPU the
final state and the inner loss of a rule run must equal the prefix-rule run
bit for bit; the outputs follow the oracle within the path's tolerance.
"""
import numpy as np
import pytest
import torch

import test_weight_sequence_ttt_b300 as ttt
from test_weight_sequence_ttt_b300.inputs import WORKLOADS, make_inputs

from _util import TOL, check_bf16_z, compare, oracle_linear, oracle_mlp, rel_err, run_linear, run_mlp, to_np

pytestmark = pytest.mark.gpu
RULES = ["anchor", "key"]

# (d, b, T, io, expected kernel kind): the split d = 64 kernel (b = 16 and b < 16
# with a ragged last super-step), the merged d = 128 kernel, the b = 64 path,
# the fp32 kernel with fp32 and with bf16 io.
LIN_CASES = [(64, 16, 48, "bf16", 2), (64, 4, 40, "bf16", 2), (64, 64, 192, "bf16", 2), (128, 16, 48, "bf16", 2),
             (128, 2, 36, "bf16", 2), (64, 256, 512, "bf16", 2), (16, 16, 64, "f32", 1), (32, 16, 48, "bf16", 1)]


def _lin(d, b, T, io, B=2, H=3, seed=123):
    w = WORKLOADS["linear_b8h12_d64_t2k"].with_(B=B, H=H, T=T, d=d, b=b, io=io, seed=seed)
    return make_inputs(w)


@pytest.mark.parametrize("rule", RULES)
@pytest.mark.parametrize("d,b,T,io,kind", LIN_CASES)
def test_linear_rule_vs_oracle(rule, d, b, T, io, kind, linear_form):
    assert ttt.linear_kernel_kind(ttt.BF16 if io == "bf16" else ttt.F32, d, b) == kind
    inp = _lin(d, b, T, io)
    got = run_linear(inp, rule=rule, q_none=rule == "key")
    assert int(got["status"].item()) == 0
    ref = oracle_linear(inp, rule=rule)
    compare(got, ref, ("Z", "W", "c", "loss", "inner_loss"), TOL[io])
    base = run_linear(inp)
    for k in ("W", "c", "inner_loss"):
        assert torch.equal(got[k], base[k]), k
    assert rel_err(to_np(got["Z"]), to_np(base["Z"])) > 1e-3  # the rule does change the outputs


@pytest.mark.parametrize("rule", RULES)
@pytest.mark.parametrize("d,h,b,T,io,kind", [(64, 256, 16, 48, "bf16", 2), (16, 48, 4, 24, "f32", 1)])
def test_mlp_rule_vs_oracle(rule, d, h, b, T, io, kind, mlp_form):
    w = WORKLOADS["mlp_b4h12_d64_t8k"].with_(B=2, H=2, T=T, d=d, hidden=h, b=b, io=io, seed=124)
    assert ttt.mlp_kernel_kind(ttt.BF16 if io == "bf16" else ttt.F32, d, h, b) == kind
    inp = make_inputs(w)
    got = run_mlp(inp, rule=rule, q_none=rule == "key")
    assert int(got["status"].item()) == 0
    ref = oracle_mlp(inp, rule=rule)
    compare(got, ref, ("Z", "W1", "c1", "W2", "c2", "loss", "inner_loss"), TOL[io])
    base = run_mlp(inp)
    for k in ("W1", "c1", "W2", "c2", "inner_loss"):
        assert torch.equal(got[k], base[k]), k


def test_key_rule_loss_is_inner_loss(linear_form):
    inp = _lin(64, 16, 64, "bf16")
    got = run_linear(inp, rule="key", q_none=True)
    assert int(got["status"].item()) == 0
    assert rel_err(to_np(got["loss"]), to_np(got["inner_loss"])) <= TOL["bf16"]


def test_key_rule_equals_anchor_rule_with_keys_as_queries(linear_form):
    inp = _lin(64, 16, 48, "bf16")
    a = run_linear(inp, rule="key", q_none=True)
    inp2 = dict(inp)
    inp2["Q"] = inp["K"]
    b = run_linear(inp2, rule="anchor")
    assert int(a["status"].item()) == 0 and int(b["status"].item()) == 0
    for k in ("Z", "W", "c", "loss", "inner_loss"):
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("rule", RULES)
def test_full_size_sampled_chains_rule(rule):
    """The headline workload in the benchmark's launch configuration, sampled chains."""
    w = WORKLOADS["linear_b8h12_d64_t2k"]
    inp = make_inputs(w)
    got = run_linear(inp, rule=rule, z_dtype=torch.bfloat16)
    assert int(got["status"].item()) == 0
    sel = sorted({0, w.chains - 1, (w.chains * 5) // 11})
    ref = oracle_linear(make_inputs(w, chains=sel), rule=rule)
    idx = (np.array([c // w.H for c in sel]), np.array([c % w.H for c in sel]))
    z = to_np(got["Z"])[idx]
    check_bf16_z(z, ref["Z"].reshape(z.shape), TOL["bf16"])
    for k in ("W", "c", "loss", "inner_loss"):
        g = to_np(got[k])[idx]
        assert rel_err(g, ref[k].reshape(g.shape)) <= 5 * TOL["bf16"], k


def test_mlp_key_rule_equals_anchor_rule_with_keys_as_queries(mlp_form):
    w = WORKLOADS["mlp_b4h12_d64_t8k"].with_(B=1, H=2, T=48, seed=125)
    inp = make_inputs(w)
    a = run_mlp(inp, rule="key", q_none=True)
    inp2 = dict(inp)
    inp2["Q"] = inp["K"]
    b = run_mlp(inp2, rule="anchor")
    assert int(a["status"].item()) == 0 and int(b["status"].item()) == 0, (a["status"], b["status"])
    for k in ("Z", "W1", "c1", "W2", "c2", "loss", "inner_loss"):
        diff = (a[k] - b[k]).abs()
        assert torch.equal(a[k], b[k]), (k, float(diff.max()), diff.nonzero()[:8].tolist())
