"""The TTT-Linear backward that allocates nothing (``ttt_linear_backward_noalloc``).

Some callers cannot allocate device memory at the moment they call the
library: code with no device allocator of its own, or a program that must keep
a fixed, planned memory footprint and cannot have an allocation fail or
synchronise the device in the middle of its work. For them the library keeps
the backward's checkpoints in a static array of its own (32 MiB per GPU) instead
of a caller workspace. These tests call that entry point through the C ABI,
twice in a row on different inputs (every call shares the array and finds the
previous call's contents in it), and check each result against the workspace
entry point ``ttt_linear_backward``. Both run the same kernel with the same
launch shape and no atomics, so the results must agree bit for bit: any
difference would be leftover scratch from the earlier call leaking in. They
also check that a call too large for the array is refused before any launch.

The file name makes pytest collect it last, so a run that stops at the first
failure has run every other test before reaching it.
"""
import ctypes

import pytest
import torch

import test_weight_sequence_ttt_b300 as ttt
from test_weight_sequence_ttt_b300 import LinearBwdArgs

pytestmark = pytest.mark.gpu

OUTS = ["dQ", "dK", "dV", "deta", "dW0", "dc0", "dln_g", "dln_b"]


def _inputs(seed, B, H, T, d, dtype):
    g = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(*s, generator=g)
    x = dict(Q=r(B, H, T, d).to(dtype), K=r(B, H, T, d).to(dtype), V=r(B, H, T, d).to(dtype),
             eta=torch.rand(B, H, T, generator=g) * 0.9 + 0.1, W0=r(1, H, d, d) * (0.5 / d ** 0.5),
             c0=r(1, H, d) * 0.1, ln_g=torch.rand(H, d, generator=g) + 0.5, ln_b=r(H, d) * 0.1,
             dZ=r(B, H, T, d).to(dtype), dW_n=r(B, H, d, d) * 0.1, dc_n=r(B, H, d) * 0.1)
    return {k: v.cuda().contiguous() for k, v in x.items()}


def _call_noalloc(x, mb, status):
    """ttt_linear_backward_noalloc through the C ABI, outputs preallocated here."""
    B, H, T, d = x["K"].shape
    out = {k: torch.empty((B, H, T, d) if k in ("dQ", "dK", "dV") else (B, H, T) if k == "deta" else
                          (B, H, d, d) if k == "dW0" else (B, H, d), device="cuda") for k in OUTS}
    a = LinearBwdArgs(B=B, H=H, T=T, d=d, mb=mb, io=ttt.BF16 if x["K"].dtype == torch.bfloat16 else ttt.F32,
                      ln_eps=1e-6, w0_bstride=0, c0_bstride=0, workspace=None, workspace_bytes=0,
                      status_dev=status.data_ptr(), eta_gate=0, eta_base=1.0,
                      **{k: x[k].data_ptr() for k in ("Q", "K", "V", "eta", "W0", "c0", "ln_g", "ln_b", "dZ",
                                                       "dW_n", "dc_n")},
                      **{k: out[k].data_ptr() for k in OUTS})
    rc = ttt.lib().ttt_linear_backward_noalloc(ctypes.byref(a), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, ttt.status_string(rc)
    return out


@pytest.mark.parametrize("d,dtype", [(64, torch.bfloat16), (32, torch.float32)])
def test_noalloc_backward_matches_workspace_entry_point_twice(d, dtype):
    B, H, T, mb = 2, 3, 256, 16
    assert ttt.linear_backward_workspace_bytes(B, H, T, d, mb) <= ttt.NOALLOC_SCRATCH_BYTES
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for seed in (1, 2):   # two calls in a row; the second finds the first one's scratch contents
        x = _inputs(seed * 10 + d, B, H, T, d, dtype)
        got = _call_noalloc(x, mb, st)
        ref = ttt.ttt_linear_backward(x["Q"], x["K"], x["V"], x["eta"], x["W0"], x["c0"], x["ln_g"], x["ln_b"],
                                      x["dZ"], mb=mb, dW_n=x["dW_n"], dc_n=x["dc_n"])
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        for k in OUTS:
            assert torch.equal(got[k], ref[k]), (seed, k, (got[k] - ref[k]).abs().max().item())


def test_noalloc_backward_refuses_sizes_beyond_its_scratch():
    # the headline workload's checkpoints (about 204 MB) do not fit the 32 MiB array
    assert ttt.linear_backward_workspace_bytes(8, 12, 2048, 64, 16) > ttt.NOALLOC_SCRATCH_BYTES
    a = LinearBwdArgs(B=8, H=12, T=2048, d=64, mb=16, io=ttt.BF16, ln_eps=1e-6)
    assert ttt.lib().ttt_linear_backward_noalloc(ctypes.byref(a), None) == 11  # TTT_ERR_SCRATCH
    assert "static" in ttt.status_string(11)
