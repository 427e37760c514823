"""Host-side checks of the C ABI (no GPU needed, no kernel launch).

* the library loads and exports every function include/ttt.h declares;
* the ctypes mirrors of the argument structs match the C layout (offsets
  printed by a tiny C program compiled with gcc against the header);
* validation returns the documented status codes before any CUDA work.
"""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

import test_weight_sequence_ttt_b300 as ttt
from test_weight_sequence_ttt_b300 import LinearArgs, LinearBwdArgs, MlpArgs, MlpBwdArgs
from test_weight_sequence_ttt_b300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ttt.h")


@pytest.fixture(scope="module")
def L():
    build()
    return ttt.lib()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ttt_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = _declared_functions()
    assert "ttt_linear_forward" in names and "ttt_mlp_forward" in names
    for n in names:
        assert hasattr(L, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", ttt.lib_path], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (ttt_\w+)", out))
    assert set(names) <= exported


def test_version_and_strings(L):
    assert ttt.abi_version() == 10
    for code in ttt.STATUS:
        assert len(ttt.status_string(code)) > 0
    assert ttt.status_string(999) == "unknown status"


def _c_offsets(struct_name, fields):
    prog = ["#include <stdio.h>", "#include <stddef.h>", '#include "%s"' % HEADER, "int main(void){"]
    prog.append('printf("%%zu\\n", sizeof(%s));' % struct_name)
    for f in fields:
        prog.append('printf("%%zu\\n", offsetof(%s, %s));' % (struct_name, f))
    prog.append("return 0;}")
    with tempfile.TemporaryDirectory() as td:
        c = os.path.join(td, "o.c")
        exe = os.path.join(td, "o")
        open(c, "w").write("\n".join(prog))
        subprocess.check_call(["gcc", "-std=c99", "-o", exe, c])
        vals = [int(x) for x in subprocess.check_output([exe]).split()]
    return vals[0], vals[1:]


@pytest.mark.parametrize("cls,cname", [(LinearArgs, "ttt_linear_args"), (MlpArgs, "ttt_mlp_args"),
                                       (LinearBwdArgs, "ttt_linear_bwd_args"), (MlpBwdArgs, "ttt_mlp_bwd_args")])
def test_struct_layout_matches_header(cls, cname):
    fields = [f[0] for f in cls._fields_]
    size, offs = _c_offsets(cname, fields)
    assert ctypes.sizeof(cls) == size
    assert [getattr(cls, f).offset for f in fields] == offs


def test_kernel_kind_table(L):
    assert ttt.linear_kernel_kind(ttt.BF16, 64, 16) == 2
    assert ttt.linear_kernel_kind(ttt.BF16, 128, 1) == 2
    assert ttt.linear_kernel_kind(ttt.BF16, 128, 64) == 2
    assert ttt.linear_kernel_kind(ttt.BF16, 64, 32) == 2
    assert ttt.linear_kernel_kind(ttt.BF16, 128, 128) == 2    # large mini-batches up to 1024
    assert ttt.linear_kernel_kind(ttt.BF16, 64, 1024) == 2
    assert ttt.linear_kernel_kind(ttt.BF16, 64, 2048) == 0    # no kernel past 1024
    assert ttt.linear_kernel_kind(ttt.BF16, 64, 96) == 0      # not a power of two, past the fp32 kernel's 64
    assert ttt.linear_kernel_kind(ttt.BF16, 64, 3) == 1       # fp32 kernel
    assert ttt.linear_kernel_kind(ttt.F32, 16, 16) == 1
    assert ttt.linear_kernel_kind(ttt.F32, 256, 16) == 0
    assert ttt.linear_kernel_kind(7, 64, 16) == 0
    assert ttt.mlp_kernel_kind(ttt.BF16, 64, 256, 16) >= 1


def _linear(**kw):
    """Well-formed argument struct with fake, 16-byte aligned, disjoint pointers."""
    B, H, T, d = kw.pop("B", 2), kw.pop("H", 3), kw.pop("T", 32), kw.pop("d", 64)
    base = 1 << 40
    step = 1 << 32
    ptrs = {n: base + i * step for i, n in enumerate(
        ["Q", "K", "V", "eta", "W0", "c0", "ln_g", "ln_b", "Z", "W_out", "c_out", "loss",
         "inner_loss", "status_dev"])}
    a = dict(B=B, H=H, T=T, d=d, mb=16, io=ttt.BF16, ln_eps=1e-6, w0_bstride=0, c0_bstride=0, **ptrs)
    a.update(kw)
    return LinearArgs(**a)


def _call(L, a):
    return L.ttt_linear_forward(ctypes.byref(a), None)


def test_validation_codes(L):
    assert L.ttt_linear_forward(None, None) == 1
    assert _call(L, _linear(Q=None)) == 1
    assert _call(L, _linear(Z=None)) == 1
    assert _call(L, _linear(T=30)) == 2                   # T % mb
    assert _call(L, _linear(T=30, partial_tail=1)) == 5   # allowed with a partial tail
    assert _call(L, _linear(partial_tail=2)) == 2
    assert _call(L, _linear(eta_gate=1, eta_base=-1.0)) == 2   # gate scale must be >= 0
    assert _call(L, _linear(eta_gate=1, eta_base=float("nan"))) == 2
    assert _call(L, _linear(eta_gate=2)) == 2
    assert _call(L, _linear(eta_gate=1, eta_base=0.5)) == 5
    assert _call(L, _linear(B=0)) == 2
    assert _call(L, _linear(ln_eps=-1.0)) == 2
    assert _call(L, _linear(w0_bstride=-4)) == 2
    assert _call(L, _linear(io=5)) == 3
    assert _call(L, _linear(d=256)) == 3
    assert _call(L, _linear(K=(1 << 40) + 3)) == 4        # misaligned
    assert _call(L, _linear(w0_bstride=6)) == 4           # stride not 16-byte multiple
    assert _call(L, _linear(Z=(1 << 40) + (1 << 32) * 1)) == 9   # Z over K
    assert _call(L, _linear(loss=(1 << 40) + (1 << 32) * 12)) == 9  # loss over inner_loss
    # well-formed, but the pointers are not device memory (no device here)
    assert _call(L, _linear()) == 5
    # output rule: out of range -> unsupported; Q may be NULL only under the key rule
    assert _call(L, _linear(out_rule=3)) == 3
    assert _call(L, _linear(out_rule=-1)) == 3
    assert _call(L, _linear(Q=None, out_rule=1)) == 1
    assert _call(L, _linear(Q=None, out_rule=2)) == 5


def test_validation_codes_mlp(L):
    base = 1 << 40
    step = 1 << 32
    names = ["Q", "K", "V", "eta", "W1_0", "c1_0", "W2_0", "c2_0", "ln_g", "ln_b", "Z", "W1_out",
             "c1_out", "W2_out", "c2_out", "loss", "inner_loss", "status_dev"]
    ptrs = {n: base + i * step for i, n in enumerate(names)}

    def call(**kw):
        a = dict(B=1, H=2, T=32, d=64, hidden=256, mb=16, io=ttt.BF16, ln_eps=1e-6, w_bstride=0,
                 c1_bstride=0, c2_bstride=0, **ptrs)
        a.update(kw)
        return L.ttt_mlp_forward(ctypes.byref(MlpArgs(**a)), None)

    assert call(W2_0=None) == 1
    assert call(T=33) == 2
    assert call(T=33, partial_tail=1) == 5
    assert call(hidden=0) == 2
    assert call(io=3) == 3
    assert call(c2_0=base + 7 * step + 4) == 4
    assert call(W1_out=base + 5 * step) == 9
    assert call() == 5
    assert call(out_rule=7) == 3
    assert call(Q=None, out_rule=0) == 1
    assert call(Q=None, out_rule=2) == 5


def test_backward_workspace_bytes(L):
    # one (W, c) anchor per mini-batch and chain, fp32
    # one (W, c) starting state per mini-batch and chain, and each token's key side, fp32
    assert ttt.linear_backward_workspace_bytes(8, 12, 2048, 64, 16) == \
        8 * 12 * (128 * (64 * 64 + 64) + 2048 * (3 * 64 + 2)) * 4
    assert ttt.linear_backward_workspace_bytes(1, 1, 16, 16, 16) == (256 + 16 + 16 * (48 + 2)) * 4
    assert ttt.linear_backward_workspace_bytes(1, 1, 30, 16, 16) == 0   # T % mb
    assert ttt.linear_backward_workspace_bytes(0, 1, 16, 16, 16) == 0


def test_validation_codes_backward(L):
    base = 1 << 40
    step = 1 << 32
    names = ["Q", "K", "V", "eta", "W0", "c0", "ln_g", "ln_b", "dZ", "dW_n", "dc_n", "dQ", "dK", "dV",
             "deta", "dW0", "dc0", "dln_g", "dln_b", "workspace", "status_dev"]
    ptrs = {n: base + i * step for i, n in enumerate(names)}
    ws = ttt.linear_backward_workspace_bytes(2, 3, 32, 64, 16)

    def call(**kw):
        a = dict(B=2, H=3, T=32, d=64, mb=16, io=ttt.BF16, ln_eps=1e-6, w0_bstride=0, c0_bstride=0,
                 workspace_bytes=ws, **ptrs)
        a.update(kw)
        return L.ttt_linear_backward(ctypes.byref(LinearBwdArgs(**a)), None)

    assert L.ttt_linear_backward(None, None) == 1
    assert call(dZ=None) == 1
    assert call(dK=None) == 1
    assert call(workspace=None) == 1
    assert call(dW_n=None, dc_n=None) == 5       # seeds are optional
    assert call(T=30) == 2                       # T % mb
    assert call(workspace_bytes=ws - 4) == 2     # workspace too small
    assert call(eta_gate=1, eta_base=-2.0) == 2
    assert call(io=4) == 3
    assert call(d=256) == 3
    assert call(mb=128, T=256) == 3
    assert call(dQ=base + 11 * step + 8) == 4    # misaligned
    assert call(dQ=base + 1 * step) == 9         # dQ over K
    assert call(workspace=base + 18 * step) == 9   # workspace over dln_b
    assert call() == 5                           # well formed; not device memory here


def test_mlp_backward_workspace_and_validation(L):
    hd = 256 * 64
    assert ttt.mlp_backward_workspace_bytes(4, 12, 8192, 64, 256, 16) == \
        48 * (512 * (2 * hd + 256 + 64) + 2 * hd + 8192 * (2 * 256 + 3 * 64 + 2)) * 4
    assert ttt.mlp_backward_workspace_bytes(1, 1, 30, 64, 256, 16) == 0
    base = 1 << 40
    step = 1 << 32
    names = ["Q", "K", "V", "eta", "W1_0", "c1_0", "W2_0", "c2_0", "ln_g", "ln_b", "dZ", "dW1_n", "dc1_n",
             "dW2_n", "dc2_n", "dQ", "dK", "dV", "deta", "dW1", "dc1", "dW2", "dc2", "dln_g", "dln_b", "workspace",
             "status_dev"]
    ptrs = {n: base + i * step for i, n in enumerate(names)}
    ws = ttt.mlp_backward_workspace_bytes(1, 2, 32, 64, 256, 16)

    def call(**kw):
        a = dict(B=1, H=2, T=32, d=64, hidden=256, mb=16, io=ttt.BF16, ln_eps=1e-6, w_bstride=0, c1_bstride=0,
                 c2_bstride=0, workspace_bytes=ws, **ptrs)
        a.update(kw)
        return L.ttt_mlp_backward(ctypes.byref(MlpBwdArgs(**a)), None)

    assert L.ttt_mlp_backward(None, None) == 1
    assert call(dW2=None) == 1
    assert call(dW1_n=None, dc1_n=None, dW2_n=None, dc2_n=None) == 5
    assert call(T=33) == 2
    assert call(workspace_bytes=ws - 16) == 2
    assert call(mb=32, T=64) == 3          # mini-batches up to 16
    assert call(d=62) == 3                 # d a multiple of 4
    assert call(dK=base + 16 * step + 4) == 4
    assert call(dW1=base + 5 * step) == 9  # dW1 over c1_0
    assert call() == 5
