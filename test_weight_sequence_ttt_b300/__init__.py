"""TTT inner loop (TTT-Linear / TTT-MLP) on one NVIDIA B300.

Thin binding over the C ABI of ``include/ttt.h`` (``libttt_b300.so``, built by
``python -m test_weight_sequence_ttt_b300.build``). This module only marshals
arguments: every step of the inner loop runs in the library's CUDA kernels.
PyTorch supplies device memory and streams.

    from test_weight_sequence_ttt_b300 import ttt_linear_forward
    out = ttt_linear_forward(Q, K, V, eta, W0, c0, ln_g, ln_b, mb=16)
    out["Z"], out["W"], out["c"], out["loss"], out["inner_loss"]
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

__all__ = [
    "TTTError", "lib", "lib_path", "ttt_linear_forward", "ttt_mlp_forward", "ttt_linear_backward",
    "linear_backward_workspace_bytes", "ttt_mlp_backward", "mlp_backward_workspace_bytes", "MlpBwdArgs",
    "status_string", "abi_version", "linear_kernel_kind", "linear_cluster_mode",
    "mlp_cluster_mode",
    "mlp_kernel_kind", "LinearArgs", "MlpArgs", "LinearBwdArgs", "STATUS", "F32", "BF16", "OUT_RULES",
    "BWD_MATH",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_HERE, "libttt_b300.so")

F32, BF16 = 0, 1
# ttt_out_rule: which weights / input produce z_t (see include/ttt.h)
OUT_RULES = {"prefix": 0, "anchor": 1, "key": 2}
# ttt_bwd_math: arithmetic of the backward's contractions (see include/ttt.h)
BWD_MATH = {"fp32": 0, "tf32": 1}
STATUS = {
    0: "TTT_OK", 1: "TTT_ERR_NULL", 2: "TTT_ERR_SHAPE", 3: "TTT_ERR_UNSUPPORTED", 4: "TTT_ERR_ALIGN",
    5: "TTT_ERR_NOT_DEVICE_PTR", 6: "TTT_ERR_CUDA", 7: "TTT_ERR_TIMEOUT", 8: "TTT_ERR_NONFINITE",
    9: "TTT_ERR_ALIAS", 10: "TTT_ERR_RANGE", 11: "TTT_ERR_SCRATCH",
}
# bytes of the library's static scratch behind ttt_linear_backward_noalloc (include/ttt.h)
NOALLOC_SCRATCH_BYTES = 32 << 20

_vp = ctypes.c_void_p


class LinearArgs(ctypes.Structure):
    """Mirror of ``ttt_linear_args``."""
    _fields_ = [
        ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("T", ctypes.c_int32), ("d", ctypes.c_int32),
        ("mb", ctypes.c_int32), ("io", ctypes.c_int32), ("z_io", ctypes.c_int32),
        ("ln_eps", ctypes.c_float),
        ("Q", _vp), ("K", _vp), ("V", _vp), ("eta", _vp), ("W0", _vp), ("c0", _vp),
        ("w0_bstride", ctypes.c_int64), ("c0_bstride", ctypes.c_int64),
        ("ln_g", _vp), ("ln_b", _vp), ("Z", _vp), ("W_out", _vp), ("c_out", _vp),
        ("loss", _vp), ("inner_loss", _vp), ("status_dev", _vp), ("out_rule", ctypes.c_int32),
        ("partial_tail", ctypes.c_int32), ("eta_gate", ctypes.c_int32), ("eta_base", ctypes.c_float),
    ]


class MlpArgs(ctypes.Structure):
    """Mirror of ``ttt_mlp_args``."""
    _fields_ = [
        ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("T", ctypes.c_int32), ("d", ctypes.c_int32),
        ("hidden", ctypes.c_int32), ("mb", ctypes.c_int32), ("io", ctypes.c_int32),
        ("z_io", ctypes.c_int32), ("ln_eps", ctypes.c_float),
        ("Q", _vp), ("K", _vp), ("V", _vp), ("eta", _vp),
        ("W1_0", _vp), ("c1_0", _vp), ("W2_0", _vp), ("c2_0", _vp),
        ("w_bstride", ctypes.c_int64), ("c1_bstride", ctypes.c_int64), ("c2_bstride", ctypes.c_int64),
        ("ln_g", _vp), ("ln_b", _vp), ("Z", _vp),
        ("W1_out", _vp), ("c1_out", _vp), ("W2_out", _vp), ("c2_out", _vp),
        ("loss", _vp), ("inner_loss", _vp), ("status_dev", _vp), ("out_rule", ctypes.c_int32),
        ("partial_tail", ctypes.c_int32), ("eta_gate", ctypes.c_int32), ("eta_base", ctypes.c_float),
    ]


class LinearBwdArgs(ctypes.Structure):
    """Mirror of ``ttt_linear_bwd_args``."""
    _fields_ = [
        ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("T", ctypes.c_int32), ("d", ctypes.c_int32),
        ("mb", ctypes.c_int32), ("io", ctypes.c_int32), ("ln_eps", ctypes.c_float),
        ("Q", _vp), ("K", _vp), ("V", _vp), ("eta", _vp), ("W0", _vp), ("c0", _vp),
        ("w0_bstride", ctypes.c_int64), ("c0_bstride", ctypes.c_int64),
        ("ln_g", _vp), ("ln_b", _vp), ("dZ", _vp), ("dW_n", _vp), ("dc_n", _vp),
        ("dQ", _vp), ("dK", _vp), ("dV", _vp), ("deta", _vp), ("dW0", _vp), ("dc0", _vp),
        ("dln_g", _vp), ("dln_b", _vp), ("workspace", _vp), ("workspace_bytes", ctypes.c_uint64),
        ("status_dev", _vp), ("eta_gate", ctypes.c_int32), ("eta_base", ctypes.c_float),
        ("math", ctypes.c_int32),
    ]


class MlpBwdArgs(ctypes.Structure):
    """Mirror of ``ttt_mlp_bwd_args``."""
    _fields_ = [
        ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("T", ctypes.c_int32), ("d", ctypes.c_int32),
        ("hidden", ctypes.c_int32), ("mb", ctypes.c_int32), ("io", ctypes.c_int32), ("ln_eps", ctypes.c_float),
        ("Q", _vp), ("K", _vp), ("V", _vp), ("eta", _vp),
        ("W1_0", _vp), ("c1_0", _vp), ("W2_0", _vp), ("c2_0", _vp),
        ("w_bstride", ctypes.c_int64), ("c1_bstride", ctypes.c_int64), ("c2_bstride", ctypes.c_int64),
        ("ln_g", _vp), ("ln_b", _vp), ("dZ", _vp),
        ("dW1_n", _vp), ("dc1_n", _vp), ("dW2_n", _vp), ("dc2_n", _vp),
        ("dQ", _vp), ("dK", _vp), ("dV", _vp), ("deta", _vp),
        ("dW1", _vp), ("dc1", _vp), ("dW2", _vp), ("dc2", _vp), ("dln_g", _vp), ("dln_b", _vp),
        ("workspace", _vp), ("workspace_bytes", ctypes.c_uint64),
        ("status_dev", _vp), ("eta_gate", ctypes.c_int32), ("eta_base", ctypes.c_float),
    ]


def _rule_code(rule) -> int:
    if isinstance(rule, str):
        if rule not in OUT_RULES:
            raise ValueError("out_rule must be one of %s" % sorted(OUT_RULES))
        return OUT_RULES[rule]
    return int(rule)


class TTTError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        msg = "%s (%d): %s" % (STATUS.get(code, "?"), code, status_string(code))
        super().__init__(msg + (" [%s]" % what if what else ""))


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """Load ``libttt_b300.so``. Raises if it has not been built: there is no
    fallback path."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(lib_path):
                raise RuntimeError(
                    "libttt_b300.so is missing; build it with "
                    "`python -m test_weight_sequence_ttt_b300.build`")
            L = ctypes.CDLL(lib_path)
            L.ttt_linear_forward.restype = ctypes.c_int
            L.ttt_linear_forward.argtypes = [ctypes.POINTER(LinearArgs), _vp]
            L.ttt_mlp_forward.restype = ctypes.c_int
            L.ttt_mlp_forward.argtypes = [ctypes.POINTER(MlpArgs), _vp]
            L.ttt_status_string.restype = ctypes.c_char_p
            L.ttt_status_string.argtypes = [ctypes.c_int]
            L.ttt_abi_version.restype = ctypes.c_int
            L.ttt_linear_cluster_mode.restype = ctypes.c_int32
            L.ttt_linear_cluster_mode.argtypes = [ctypes.c_int32]
            L.ttt_mlp_cluster_mode.restype = ctypes.c_int32
            L.ttt_mlp_cluster_mode.argtypes = [ctypes.c_int32]
            L.ttt_abi_version.argtypes = []
            L.ttt_linear_kernel_kind.restype = ctypes.c_int
            L.ttt_linear_kernel_kind.argtypes = [ctypes.c_int32] * 3
            L.ttt_mlp_kernel_kind.restype = ctypes.c_int
            L.ttt_mlp_kernel_kind.argtypes = [ctypes.c_int32] * 4
            L.ttt_linear_backward.restype = ctypes.c_int
            L.ttt_linear_backward.argtypes = [ctypes.POINTER(LinearBwdArgs), _vp]
            L.ttt_linear_backward_workspace_bytes.restype = ctypes.c_uint64
            L.ttt_linear_backward_workspace_bytes.argtypes = [ctypes.c_int32] * 5
            L.ttt_linear_backward_noalloc.restype = ctypes.c_int
            L.ttt_linear_backward_noalloc.argtypes = [ctypes.POINTER(LinearBwdArgs), _vp]
            L.ttt_mlp_backward.restype = ctypes.c_int
            L.ttt_mlp_backward.argtypes = [ctypes.POINTER(MlpBwdArgs), _vp]
            L.ttt_mlp_backward_workspace_bytes.restype = ctypes.c_uint64
            L.ttt_mlp_backward_workspace_bytes.argtypes = [ctypes.c_int32] * 6
            _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().ttt_status_string(int(code)).decode()


def abi_version() -> int:
    return lib().ttt_abi_version()


def linear_cluster_mode(mode: int = -1) -> int:
    """Set (0 never, the default; 1 when 2 * B * H <= SMs; 2 always) and
    return the form of the d = 64,
    mb = 16 TTT-Linear kernel that runs each chain on a two-CTA cluster; any
    other value only reads the current mode (see include/ttt.h)."""
    return int(lib().ttt_linear_cluster_mode(int(mode)))


def mlp_cluster_mode(mode: int = -1) -> int:
    """Set (0 never; 1 when 2 * B * H <= SMs, the default; 2 always) and
    return the form of the tensor-core TTT-MLP kernel that runs each chain on
    a two-CTA cluster with the hidden units split; any other value only reads
    the current mode (see include/ttt.h)."""
    return int(lib().ttt_mlp_cluster_mode(int(mode)))


def linear_kernel_kind(io: int, d: int, mb: int) -> int:
    return lib().ttt_linear_kernel_kind(io, d, mb)


def mlp_kernel_kind(io: int, d: int, hidden: int, mb: int) -> int:
    return lib().ttt_mlp_kernel_kind(io, d, hidden, mb)


# ---------------------------------------------------------------- marshalling helpers

def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _io_code(dtype) -> int:
    import torch
    if dtype == torch.float32:
        return F32
    if dtype == torch.bfloat16:
        return BF16
    raise TypeError("Q/K/V must be float32 or bfloat16, got %s" % dtype)


def _check_cuda(name, t):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def _bstride(t, B: int, per: int) -> int:
    if t.shape[0] == 1:
        return 0 if B > 1 else per
    if t.shape[0] != B:
        raise ValueError("initial weights need a leading dim of B or 1")
    return per


def _stream_handle(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def ttt_linear_forward(Q, K, V, eta, W0, c0, ln_g, ln_b, *, mb: int, eps: float = 1e-6,
                       z_dtype=None, out: Optional[dict] = None, want_state: bool = True,
                       want_loss: bool = True, want_inner_loss: bool = True,
                       status=None, stream=None, out_rule="prefix", partial_tail: bool = False,
                       eta_gate: bool = False, eta_base: float = 1.0) -> dict:
    """Run the TTT-Linear inner loop through ``ttt_linear_forward``.

    Q, K, V [B,H,T,d] (float32 or bfloat16, CUDA, contiguous); eta [B,H,T] fp32;
    W0 [B|1,H,d,d], c0 [B|1,H,d], ln_g/ln_b [H,d] fp32. ``out`` may pass
    preallocated outputs (keys Z, W, c, loss, inner_loss); missing ones are
    allocated with torch. ``z_dtype`` (torch.float32 by default, or
    torch.bfloat16) is the element type of Z; a preallocated Z sets it. ``status`` is an optional int32 CUDA tensor of one
    element (0 on entry) that receives device-side errors. Asynchronous on
    ``stream`` (default: torch's current stream). ``out_rule`` is "prefix"
    (z_t = f(q_t; W_t)), "anchor" (z_t = f(q_t; W_{i-1})) or "key"
    (z_t = f(k_t; W_{i-1}); Q may be None). ``partial_tail`` lets T % mb != 0:
    the last T % mb tokens are emitted but not committed (W, c stay at the
    state after the last full mini-batch). With ``eta_gate`` the ``eta``
    argument holds the gate logits theta_lr . x and the kernels compute
    eta = eta_base * sigmoid(logit)."""
    import torch
    rule = _rule_code(out_rule)
    for n, t in (("Q", Q), ("K", K), ("V", V), ("eta", eta), ("W0", W0), ("c0", c0),
                 ("ln_g", ln_g), ("ln_b", ln_b), ("status", status)):
        _check_cuda(n, t)
    B, H, T, d = K.shape
    out = dict(out or {})
    dev = K.device
    if "Z" not in out:
        out["Z"] = torch.empty(K.shape, device=dev, dtype=z_dtype or torch.float32)
    if want_state:
        out.setdefault("W", torch.empty(B, H, d, d, device=dev, dtype=torch.float32))
        out.setdefault("c", torch.empty(B, H, d, device=dev, dtype=torch.float32))
    if want_loss:
        out.setdefault("loss", torch.empty(B, H, T, device=dev, dtype=torch.float32))
    if want_inner_loss:
        out.setdefault("inner_loss", torch.empty(B, H, T, device=dev, dtype=torch.float32))
    a = LinearArgs(
        B=B, H=H, T=T, d=d, mb=mb, io=_io_code(K.dtype), z_io=_io_code(out["Z"].dtype), ln_eps=eps,
        Q=_ptr(Q), K=_ptr(K), V=_ptr(V), eta=_ptr(eta), W0=_ptr(W0), c0=_ptr(c0),
        w0_bstride=_bstride(W0, B, H * d * d), c0_bstride=_bstride(c0, B, H * d),
        ln_g=_ptr(ln_g), ln_b=_ptr(ln_b), Z=_ptr(out["Z"]), W_out=_ptr(out.get("W")),
        c_out=_ptr(out.get("c")), loss=_ptr(out.get("loss")),
        inner_loss=_ptr(out.get("inner_loss")), status_dev=_ptr(status), out_rule=rule,
        partial_tail=int(bool(partial_tail)), eta_gate=int(bool(eta_gate)), eta_base=float(eta_base),
    )
    rc = lib().ttt_linear_forward(ctypes.byref(a), _stream_handle(stream))
    if rc != 0:
        raise TTTError(rc, "ttt_linear_forward")
    return out


def ttt_mlp_forward(Q, K, V, eta, W1, c1, W2, c2, ln_g, ln_b, *, mb: int, eps: float = 1e-6,
                    z_dtype=None, out: Optional[dict] = None, want_state: bool = True,
                    want_loss: bool = True, want_inner_loss: bool = True,
                    status=None, stream=None, out_rule="prefix", partial_tail: bool = False,
                    eta_gate: bool = False, eta_base: float = 1.0) -> dict:
    """Run the TTT-MLP inner loop through ``ttt_mlp_forward``.

    W1 [B|1,H,h,d], c1 [B|1,H,h], W2 [B|1,H,d,h], c2 [B|1,H,d] fp32; other
    arguments as for ``ttt_linear_forward``. Outputs: Z, W1, c1, W2, c2, loss,
    inner_loss."""
    import torch
    rule = _rule_code(out_rule)
    for n, t in (("Q", Q), ("K", K), ("V", V), ("eta", eta), ("W1", W1), ("c1", c1), ("W2", W2),
                 ("c2", c2), ("ln_g", ln_g), ("ln_b", ln_b), ("status", status)):
        _check_cuda(n, t)
    B, H, T, d = K.shape
    h = W1.shape[-2]
    out = dict(out or {})
    dev = K.device
    if "Z" not in out:
        out["Z"] = torch.empty(K.shape, device=dev, dtype=z_dtype or torch.float32)
    if want_state:
        out.setdefault("W1", torch.empty(B, H, h, d, device=dev, dtype=torch.float32))
        out.setdefault("c1", torch.empty(B, H, h, device=dev, dtype=torch.float32))
        out.setdefault("W2", torch.empty(B, H, d, h, device=dev, dtype=torch.float32))
        out.setdefault("c2", torch.empty(B, H, d, device=dev, dtype=torch.float32))
    if want_loss:
        out.setdefault("loss", torch.empty(B, H, T, device=dev, dtype=torch.float32))
    if want_inner_loss:
        out.setdefault("inner_loss", torch.empty(B, H, T, device=dev, dtype=torch.float32))
    a = MlpArgs(
        B=B, H=H, T=T, d=d, hidden=h, mb=mb, io=_io_code(K.dtype), z_io=_io_code(out["Z"].dtype),
        ln_eps=eps,
        Q=_ptr(Q), K=_ptr(K), V=_ptr(V), eta=_ptr(eta),
        W1_0=_ptr(W1), c1_0=_ptr(c1), W2_0=_ptr(W2), c2_0=_ptr(c2),
        w_bstride=_bstride(W1, B, H * h * d), c1_bstride=_bstride(c1, B, H * h),
        c2_bstride=_bstride(c2, B, H * d),
        ln_g=_ptr(ln_g), ln_b=_ptr(ln_b), Z=_ptr(out["Z"]),
        W1_out=_ptr(out.get("W1")), c1_out=_ptr(out.get("c1")), W2_out=_ptr(out.get("W2")),
        c2_out=_ptr(out.get("c2")), loss=_ptr(out.get("loss")),
        inner_loss=_ptr(out.get("inner_loss")), status_dev=_ptr(status), out_rule=rule,
        partial_tail=int(bool(partial_tail)), eta_gate=int(bool(eta_gate)), eta_base=float(eta_base),
    )
    rc = lib().ttt_mlp_forward(ctypes.byref(a), _stream_handle(stream))
    if rc != 0:
        raise TTTError(rc, "ttt_mlp_forward")
    return out


def linear_backward_workspace_bytes(B: int, H: int, T: int, d: int, mb: int) -> int:
    """Device scratch ``ttt_linear_backward`` needs (0 for invalid sizes)."""
    return int(lib().ttt_linear_backward_workspace_bytes(B, H, T, d, mb))


def ttt_linear_backward(Q, K, V, eta, W0, c0, ln_g, ln_b, dZ, *, mb: int, dW_n=None, dc_n=None,
                        eps: float = 1e-6, out: Optional[dict] = None, workspace=None, status=None,
                        stream=None, eta_gate: bool = False, eta_base: float = 1.0, math: str = "fp32") -> dict:
    """Gradients of the TTT-Linear inner loop through ``ttt_linear_backward``.

    Inputs as for ``ttt_linear_forward`` (prefix rule, T a multiple of mb)
    plus dZ [B,H,T,d] in the dtype of Q/K/V and optional final-state seeds
    dW_n [B,H,d,d], dc_n [B,H,d] fp32. Returns fp32 dQ, dK, dV [B,H,T,d], deta
    [B,H,T] (w.r.t. the gate logits with ``eta_gate``) and per-chain dW0
    [B,H,d,d], dc0, dln_g, dln_b [B,H,d] (sum over B for parameters shared by
    the sequences). ``workspace`` is an optional uint8 CUDA tensor of at least
    ``linear_backward_workspace_bytes`` bytes; one is allocated otherwise.
    ``math`` is "fp32" (every product in fp32) or "tf32" (for d = 64, mb = 16
    the products run on the tensor cores with tf32 operands; include/ttt.h)."""
    import torch
    if math not in BWD_MATH:
        raise ValueError("math must be one of %s" % sorted(BWD_MATH))
    for n, t in (("Q", Q), ("K", K), ("V", V), ("eta", eta), ("W0", W0), ("c0", c0), ("ln_g", ln_g),
                 ("ln_b", ln_b), ("dZ", dZ), ("dW_n", dW_n), ("dc_n", dc_n), ("workspace", workspace),
                 ("status", status)):
        _check_cuda(n, t)
    if dZ.dtype != K.dtype:
        raise TypeError("dZ must have the dtype of Q/K/V")
    B, H, T, d = K.shape
    dev = K.device
    out = dict(out or {})
    f32 = dict(device=dev, dtype=torch.float32)
    for k, shape in (("dQ", (B, H, T, d)), ("dK", (B, H, T, d)), ("dV", (B, H, T, d)), ("deta", (B, H, T)),
                     ("dW0", (B, H, d, d)), ("dc0", (B, H, d)), ("dln_g", (B, H, d)), ("dln_b", (B, H, d))):
        if k not in out:
            out[k] = torch.empty(shape, **f32)
    need = linear_backward_workspace_bytes(B, H, T, d, mb)
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=dev, dtype=torch.uint8)
    a = LinearBwdArgs(
        B=B, H=H, T=T, d=d, mb=mb, io=_io_code(K.dtype), ln_eps=eps,
        Q=_ptr(Q), K=_ptr(K), V=_ptr(V), eta=_ptr(eta), W0=_ptr(W0), c0=_ptr(c0),
        w0_bstride=_bstride(W0, B, H * d * d), c0_bstride=_bstride(c0, B, H * d),
        ln_g=_ptr(ln_g), ln_b=_ptr(ln_b), dZ=_ptr(dZ), dW_n=_ptr(dW_n), dc_n=_ptr(dc_n),
        dQ=_ptr(out["dQ"]), dK=_ptr(out["dK"]), dV=_ptr(out["dV"]), deta=_ptr(out["deta"]),
        dW0=_ptr(out["dW0"]), dc0=_ptr(out["dc0"]), dln_g=_ptr(out["dln_g"]), dln_b=_ptr(out["dln_b"]),
        workspace=_ptr(workspace), workspace_bytes=workspace.numel() * workspace.element_size(),
        status_dev=_ptr(status), eta_gate=int(bool(eta_gate)), eta_base=float(eta_base),
        math=BWD_MATH[math],
    )
    rc = lib().ttt_linear_backward(ctypes.byref(a), _stream_handle(stream))
    if rc != 0:
        raise TTTError(rc, "ttt_linear_backward")
    return out


def mlp_backward_workspace_bytes(B: int, H: int, T: int, d: int, hidden: int, mb: int) -> int:
    """Device scratch ``ttt_mlp_backward`` needs (0 for invalid sizes)."""
    return int(lib().ttt_mlp_backward_workspace_bytes(B, H, T, d, hidden, mb))


def ttt_mlp_backward(Q, K, V, eta, W1, c1, W2, c2, ln_g, ln_b, dZ, *, mb: int, dW1_n=None, dc1_n=None,
                     dW2_n=None, dc2_n=None, eps: float = 1e-6, out: Optional[dict] = None, workspace=None,
                     status=None, stream=None, eta_gate: bool = False, eta_base: float = 1.0) -> dict:
    """Gradients of the TTT-MLP inner loop through ``ttt_mlp_backward``.

    Inputs as for ``ttt_mlp_forward`` (prefix rule, T a multiple of mb) plus dZ
    in the dtype of Q/K/V and optional fp32 final-state seeds. Returns fp32 dQ,
    dK, dV, deta and per-chain dW1, dc1, dW2, dc2, dln_g, dln_b."""
    import torch
    for n, t in (("Q", Q), ("K", K), ("V", V), ("eta", eta), ("W1", W1), ("c1", c1), ("W2", W2), ("c2", c2),
                 ("ln_g", ln_g), ("ln_b", ln_b), ("dZ", dZ), ("dW1_n", dW1_n), ("dc1_n", dc1_n),
                 ("dW2_n", dW2_n), ("dc2_n", dc2_n), ("workspace", workspace), ("status", status)):
        _check_cuda(n, t)
    if dZ.dtype != K.dtype:
        raise TypeError("dZ must have the dtype of Q/K/V")
    B, H, T, d = K.shape
    h = W1.shape[-2]
    dev = K.device
    out = dict(out or {})
    f32 = dict(device=dev, dtype=torch.float32)
    for k, shape in (("dQ", (B, H, T, d)), ("dK", (B, H, T, d)), ("dV", (B, H, T, d)), ("deta", (B, H, T)),
                     ("dW1", (B, H, h, d)), ("dc1", (B, H, h)), ("dW2", (B, H, d, h)), ("dc2", (B, H, d)),
                     ("dln_g", (B, H, d)), ("dln_b", (B, H, d))):
        if k not in out:
            out[k] = torch.empty(shape, **f32)
    if workspace is None:
        workspace = torch.empty(max(mlp_backward_workspace_bytes(B, H, T, d, h, mb), 16), device=dev,
                                dtype=torch.uint8)
    a = MlpBwdArgs(
        B=B, H=H, T=T, d=d, hidden=h, mb=mb, io=_io_code(K.dtype), ln_eps=eps,
        Q=_ptr(Q), K=_ptr(K), V=_ptr(V), eta=_ptr(eta), W1_0=_ptr(W1), c1_0=_ptr(c1), W2_0=_ptr(W2),
        c2_0=_ptr(c2), w_bstride=_bstride(W1, B, H * h * d), c1_bstride=_bstride(c1, B, H * h),
        c2_bstride=_bstride(c2, B, H * d), ln_g=_ptr(ln_g), ln_b=_ptr(ln_b), dZ=_ptr(dZ),
        dW1_n=_ptr(dW1_n), dc1_n=_ptr(dc1_n), dW2_n=_ptr(dW2_n), dc2_n=_ptr(dc2_n),
        dQ=_ptr(out["dQ"]), dK=_ptr(out["dK"]), dV=_ptr(out["dV"]), deta=_ptr(out["deta"]),
        dW1=_ptr(out["dW1"]), dc1=_ptr(out["dc1"]), dW2=_ptr(out["dW2"]), dc2=_ptr(out["dc2"]),
        dln_g=_ptr(out["dln_g"]), dln_b=_ptr(out["dln_b"]),
        workspace=_ptr(workspace), workspace_bytes=workspace.numel() * workspace.element_size(),
        status_dev=_ptr(status), eta_gate=int(bool(eta_gate)), eta_base=float(eta_base),
    )
    rc = lib().ttt_mlp_backward(ctypes.byref(a), _stream_handle(stream))
    if rc != 0:
        raise TTTError(rc, "ttt_mlp_backward")
    return out
