"""Shared helpers for the GPU parity tests (kernel vs fp64 oracle)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import test_weight_sequence_ttt_b300 as ttt

# Tolerances on max |err| relative to RMS of the oracle's tensor (over the whole
# tensor). fp32 path: 1e-4; bf16-io / fp16-operand tensor-core path: 2e-2.
TOL = {"f32": 1e-4, "bf16": 2e-2}


def rms(a) -> float:
    a = np.asarray(a, np.float64)
    return float(np.sqrt(np.mean(a * a))) if a.size else 0.0


def rel_err(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    r = rms(ref)
    return float(np.abs(got - ref).max() / (r if r > 0 else 1.0))


def to_np(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def dev(inp: dict) -> dict:
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def run_linear(inp: dict, *, status=True, out=None, z_dtype=torch.float32, rule="prefix", q_none=False):
    d = dev(inp)
    st = torch.zeros(1, dtype=torch.int32, device="cuda") if status else None
    o = ttt.ttt_linear_forward(None if q_none else d["Q"], d["K"], d["V"], d["eta"], d["W0"], d["c0"],
                               d["ln_g"], d["ln_b"], mb=inp["b"], eps=inp["eps"], status=st, out=out,
                               z_dtype=z_dtype, out_rule=rule)
    torch.cuda.synchronize()
    o["status"] = st
    return o


def run_mlp(inp: dict, *, status=True, z_dtype=torch.float32, rule="prefix", q_none=False):
    d = dev(inp)
    st = torch.zeros(1, dtype=torch.int32, device="cuda") if status else None
    o = ttt.ttt_mlp_forward(None if q_none else d["Q"], d["K"], d["V"], d["eta"], d["W1"], d["c1"], d["W2"],
                            d["c2"], d["ln_g"], d["ln_b"], mb=inp["b"], eps=inp["eps"], status=st,
                            z_dtype=z_dtype, out_rule=rule)
    torch.cuda.synchronize()
    o["status"] = st
    return o


def oracle_linear(inp: dict, nthreads: int = 0, rule: str = "prefix", partial_tail: bool = False) -> dict:
    return oracle.ttt_linear(to_np(inp["Q"]), to_np(inp["K"]), to_np(inp["V"]), to_np(inp["eta"]),
                             to_np(inp["W0"]), to_np(inp["c0"]), to_np(inp["ln_g"]), to_np(inp["ln_b"]),
                             b=inp["b"], eps=inp["eps"], nthreads=nthreads, rule=rule, partial_tail=partial_tail)


def oracle_mlp(inp: dict, nthreads: int = 0, rule: str = "prefix", partial_tail: bool = False) -> dict:
    return oracle.ttt_mlp(to_np(inp["Q"]), to_np(inp["K"]), to_np(inp["V"]), to_np(inp["eta"]),
                          to_np(inp["W1"]), to_np(inp["c1"]), to_np(inp["W2"]), to_np(inp["c2"]),
                          to_np(inp["ln_g"]), to_np(inp["ln_b"]), b=inp["b"], eps=inp["eps"],
                          nthreads=nthreads, rule=rule, partial_tail=partial_tail)


def compare(got: dict, ref: dict, keys, tol: float, sel=None) -> dict:
    """Relative max errors per output; asserts each is within ``tol``.
    ``sel`` (index tuple) restricts the kernel's outputs to sampled chains."""
    errs = {}
    for k in keys:
        g = to_np(got[k])
        if sel is not None:
            g = g[sel]
        errs[k] = rel_err(g.reshape(ref[k].shape), ref[k])
    bad = {k: e for k, e in errs.items() if not e <= tol}
    assert not bad, "max|err|/RMS above %.1e: %s (all: %s)" % (tol, bad, errs)
    return errs


BF16_HALF_ULP = 2.0 ** -8   # largest relative rounding error of a bf16 value


def check_bf16_z(z_got, z_ref, tol: float) -> float:
    """bf16 Z: every element within tol * RMS(Z) of the oracle plus the bf16
    format's own rounding bound 2^-8 |z|. Returns the arithmetic part of the
    worst error, max(|err| - 2^-8 |z_ref|) / RMS(Z)."""
    g = np.asarray(to_np(z_got) if isinstance(z_got, torch.Tensor) else z_got, np.float64)
    r = np.asarray(z_ref, np.float64).reshape(g.shape)
    R = rms(r)
    excess = (np.abs(g - r) - BF16_HALF_ULP * np.abs(r)).max() / R
    assert excess <= tol, "bf16 Z: arithmetic error %.3e * RMS(Z) above %.1e" % (excess, tol)
    return float(excess)
