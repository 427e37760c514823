"""Seeded synthetic inputs for the TTT inner loop.

This module only draws random inputs with the shapes and distributions of the
named workloads. It holds none of the inner-loop arithmetic, so both the CUDA
path and the CPU oracle can be fed from it.

Every chain (sequence beta, head h) is drawn from its own generator, seeded
from (workload seed, chain index, stream tag), so any subset of chains can be
regenerated alone -- the oracle re-derives exactly the chains it samples.

Distributions (per workload, see ``WORKLOADS``):
  * Q, K, V: N(0, 1) rounded once to the io dtype (bf16), or, for the tiny fp32
    workload, projections theta_{Q,K,V} x_t with x_t ~ N(0, I_d) and
    theta ~ N(0, 1/d) per head.
  * eta_t = eta_base * sigmoid(theta_lr . x_t), theta_lr ~ N(0, 0.02^2) per head.
    Where x_t is not otherwise drawn, theta_lr . x_t is drawn directly as
    N(0, ||theta_lr||^2): the same distribution without d extra draws per token.
  * Initial fast weights ~ N(0, 0.02^2), one set per head shared by all sequences
    (a learned W_0); biases 0; LayerNorm gamma = 1, beta = 0, eps = 1e-6.
  * Backward (``make_cotangents``): upstream gradients dZ ~ N(0, 1) rounded to
    the io dtype, final-state seeds dW_n, dc_n ~ N(0, 0.1^2) fp32.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

_TAGS = {"Q": 1, "K": 2, "V": 3, "eta": 4, "x": 5, "W0": 6, "W1": 7, "W2": 8,
         "thK": 9, "thV": 10, "thQ": 11, "thlr": 12, "dZ": 13, "dWn": 14, "dcn": 15, "dW2n": 16, "dc2n": 17}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    variant: str          # "linear" or "mlp"
    B: int
    H: int
    T: int
    d: int
    b: int
    io: str               # "f32" or "bf16"
    hidden: int = 0       # MLP hidden width (4d on the pages)
    seed: int = 0
    projected: bool = False  # Q/K/V = theta x (tiny fp32 workload) instead of N(0,1)
    eta_base: float = 1.0
    w_std: float = 0.02
    eps: float = 1e-6
    partial_tail: bool = False  # T % b tokens at the end are emitted, not committed

    @property
    def chains(self) -> int:
        return self.B * self.H

    @property
    def tokens(self) -> int:
        return self.B * self.H * self.T

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    # tiny fp32 parity case: projected x, oracle runs in milliseconds
    "linear_f32_tiny": Workload("linear_f32_tiny", "linear", 1, 1, 64, 16, 16, "f32",
                                seed=1001, projected=True),
    # TTT-Linear, 8 sequences x 12 heads, d=64, T=2K, b=16 (the headline workload)
    "linear_b8h12_d64_t2k": Workload("linear_b8h12_d64_t2k", "linear", 8, 12, 2048, 64, 16,
                                     "bf16", seed=1002),
    # TTT-MLP d=64 -> 256 -> 64, 4 x 12 chains, T=8K
    "mlp_b4h12_d64_t8k": Workload("mlp_b4h12_d64_t8k", "mlp", 4, 12, 8192, 64, 16, "bf16",
                                  hidden=256, seed=1003),
    # long-context TTT-Linear prefill, 1 x 32 chains, T=128K
    "linear_b1h32_d64_t128k": Workload("linear_b1h32_d64_t128k", "linear", 1, 32, 131072, 64,
                                       16, "bf16", seed=1004),
    # mini-batch sweep, d=128, 16 x 16 chains, T=4K (b in {1,4,16,64})
    "linear_b16h16_d128_t4k_mb1": Workload("linear_b16h16_d128_t4k_mb1", "linear", 16, 16,
                                           4096, 128, 1, "bf16", seed=1005),
    "linear_b16h16_d128_t4k_mb4": Workload("linear_b16h16_d128_t4k_mb4", "linear", 16, 16,
                                           4096, 128, 4, "bf16", seed=1005),
    "linear_b16h16_d128_t4k_mb16": Workload("linear_b16h16_d128_t4k_mb16", "linear", 16, 16,
                                            4096, 128, 16, "bf16", seed=1005),
    "linear_b16h16_d128_t4k_mb64": Workload("linear_b16h16_d128_t4k_mb64", "linear", 16, 16,
                                            4096, 128, 64, "bf16", seed=1005),
    # large mini-batch (the E2E review's b = 1K regime): the headline chains, T = 8K, b = 1024
    "linear_b8h12_d64_t8k_mb1024": Workload("linear_b8h12_d64_t8k_mb1024", "linear", 8, 12, 8192, 64, 1024,
                                            "bf16", seed=1008),
    # decode step: 15 tokens of an unfilled mini-batch per chain, emitted from the
    # committed state (the worst case before the 16th token commits the batch)
    "linear_b8h12_d64_decode15": Workload("linear_b8h12_d64_decode15", "linear", 8, 12, 15, 64, 16,
                                          "bf16", seed=1006, partial_tail=True),
    "mlp_b4h12_d64_decode15": Workload("mlp_b4h12_d64_decode15", "mlp", 4, 12, 15, 64, 16, "bf16",
                                       hidden=256, seed=1007, partial_tail=True),
}


def _gen(seed: int, chain: int, tag: str) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed((seed * 1_000_003 + chain * 101 + _TAGS[tag]) % (2 ** 63 - 1))
    return g


def _io_dtype(io: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[io]


def make_inputs(w: Workload, chains: Optional[Sequence[int]] = None) -> dict:
    """Inputs of workload ``w`` as CPU tensors.

    ``chains`` selects a subset of chain indices (beta * H + h); the result then
    has a leading chain axis of that length folded as B = len(chains), H = 1,
    with the per-head weights of each chain's head.

    Returns dict: Q, K, V [B,H,T,d] (io dtype), eta [B,H,T] fp32, LN gamma/beta
    [H,d] fp32, eps, b, and the initial weights (fp32):
      linear: W0 [1,H,d,d], c0 [1,H,d]
      mlp:    W1 [1,H,h,d], c1 [1,H,h], W2 [1,H,d,h], c2 [1,H,d]
    (subset form: initial weights [n,1,...], one per selected chain).
    """
    d, T, H = w.d, w.T, w.H
    sel = list(range(w.chains)) if chains is None else list(chains)
    dt = _io_dtype(w.io)
    Qs, Ks, Vs, etas, logits = [], [], [], [], []
    for ch in sel:
        hh = ch % H
        if w.projected:
            x = torch.randn(T, d, generator=_gen(w.seed, ch, "x"), dtype=torch.float64)
            th = {t: torch.randn(d, d, generator=_gen(w.seed, hh, t), dtype=torch.float64)
                  / math.sqrt(d) for t in ("thK", "thV", "thQ")}
            Qs.append((x @ th["thQ"].T).to(dt))
            Ks.append((x @ th["thK"].T).to(dt))
            Vs.append((x @ th["thV"].T).to(dt))
            thlr = torch.randn(d, generator=_gen(w.seed, hh, "thlr"), dtype=torch.float64) * 0.02
            u = x @ thlr
        else:
            Qs.append(torch.randn(T, d, generator=_gen(w.seed, ch, "Q")).to(dt))
            Ks.append(torch.randn(T, d, generator=_gen(w.seed, ch, "K")).to(dt))
            Vs.append(torch.randn(T, d, generator=_gen(w.seed, ch, "V")).to(dt))
            thlr = torch.randn(d, generator=_gen(w.seed, hh, "thlr"), dtype=torch.float64) * 0.02
            u = torch.randn(T, generator=_gen(w.seed, ch, "eta"), dtype=torch.float64) * thlr.norm()
        etas.append((w.eta_base * torch.sigmoid(u)).to(torch.float32))
        logits.append(u.to(torch.float32))
    if chains is None:
        shp = (w.B, H)
        heads = list(range(H))
    else:
        shp = (len(sel), 1)
        heads = [ch % H for ch in sel]
    out = dict(
        Q=torch.stack(Qs).reshape(*shp, T, d),
        K=torch.stack(Ks).reshape(*shp, T, d),
        V=torch.stack(Vs).reshape(*shp, T, d),
        eta=torch.stack(etas).reshape(*shp, T),
        eta_logit=torch.stack(logits).reshape(*shp, T),  # theta_lr . x_t, for the in-kernel gate
        b=w.b, eps=w.eps,
    )
    ln_g = torch.ones(H, d)
    ln_b = torch.zeros(H, d)

    def per_head(tag, shape):
        return torch.stack([torch.randn(*shape, generator=_gen(w.seed, hh, tag)) * w.w_std
                            for hh in heads])

    if w.variant == "linear":
        W0 = per_head("W0", (d, d))
        c0 = torch.zeros(len(heads), d)
        if chains is None:
            out.update(W0=W0[None], c0=c0[None], ln_g=ln_g, ln_b=ln_b)
        else:
            out.update(W0=W0[:, None], c0=c0[:, None], ln_g=ln_g[:1], ln_b=ln_b[:1])
    else:
        hd = w.hidden
        W1 = per_head("W1", (hd, d))
        W2 = per_head("W2", (d, hd))
        c1 = torch.zeros(len(heads), hd)
        c2 = torch.zeros(len(heads), d)
        if chains is None:
            out.update(W1=W1[None], c1=c1[None], W2=W2[None], c2=c2[None], ln_g=ln_g, ln_b=ln_b)
        else:
            out.update(W1=W1[:, None], c1=c1[:, None], W2=W2[:, None], c2=c2[:, None],
                       ln_g=ln_g[:1], ln_b=ln_b[:1])
    return out


def make_cotangents(w: Workload, chains: Optional[Sequence[int]] = None) -> dict:
    """Upstream gradients for the backward of workload ``w`` (CPU tensors):
    dZ [B,H,T,d] in the io dtype and fp32 seeds on the final state -- linear:
    dW_n [B,H,d,d], dc_n [B,H,d]; mlp: dW1_n [B,H,h,d], dc1_n [B,H,h], dW2_n
    [B,H,d,h], dc2_n [B,H,d] -- one generator per chain as in ``make_inputs``
    (same ``chains`` subset form)."""
    d, T = w.d, w.T
    sel = list(range(w.chains)) if chains is None else list(chains)
    shp = (w.B, w.H) if chains is None else (len(sel), 1)
    dt = _io_dtype(w.io)
    dZ = torch.stack([torch.randn(T, d, generator=_gen(w.seed, ch, "dZ")).to(dt) for ch in sel])
    out = dict(dZ=dZ.reshape(*shp, T, d))

    def seed(tag, shape):
        g = [_gen(w.seed, ch, tag) for ch in sel]
        return torch.stack([torch.randn(*shape, generator=gg) * 0.1 for gg in g]).reshape(*shp, *shape)

    if w.variant == "linear":
        out.update(dW_n=seed("dWn", (d, d)), dc_n=seed("dcn", (d,)))
    else:
        h = w.hidden
        out.update(dW1_n=seed("dWn", (h, d)), dc1_n=seed("dcn", (h,)), dW2_n=seed("dW2n", (d, h)),
                   dc2_n=seed("dc2n", (d,)))
    return out
