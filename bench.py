#!/usr/bin/env python
"""Benchmark of the TTT inner loop on one B300 (tokens/s and roofline fraction).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one call of the library over the whole workload (every chain, every
token): the full TTT inner loop -- loads, key forward, LayerNorm
forward/backward, in-batch mixing, output, weight update, final state.
Default workload: the long-context TTT-Linear prefill scan, 1 sequence x 32
heads, d=64, T=131072, b=16 (2.16 GB of Q/K/V/eta/Z per call: the largest of
the workloads that fit one GPU).

``--gpus N`` runs one process per GPU. Without a torchrun environment the
script starts the N processes itself (torch.distributed.run, 127.0.0.1). Every
chain is independent, so the scaling is weak: each rank runs its own seeded
workload of the same shape (its chains are distinct units of one job of N
times the chains), with no collective on the data path; rank 0 prints the
whole-job tokens/s over the slowest rank's time. ``--host-only`` replaces the
GPU step by the CPU oracle on a small slice of each rank's chains (gloo), for
testing this multi-process logic on a machine without GPUs.

Prints one JSON line. ``value`` is whole-job throughput (B*T*H tokens per
second over all ranks) with inputs resident in HBM, timed per step with CUDA
events on the launching stream and L2 flushed (256 MiB write) between steps.
``e2e`` is the same metric through the C ABI with pinned host buffers: the
host->device copies of the step's inputs and the device->host copies of all
its outputs (Z, the final state, the per-token losses) are inside the timed
region, pipelined across steps on
separate streams (inputs of step k in while step k-1 computes, results of
step k-1 out while step k computes). ``cpu_baseline`` times the
fp64 CPU oracle on a bounded sample of the same workload.

``--impl reference`` runs the reference arm: the fp64 CPU oracle as it stands,
one bounded sample of the workload per step, on the host cores.

``--backward`` times the outer-loop gradient instead: one step is one
``ttt_linear_backward`` (or, for a TTT-MLP workload, ``ttt_mlp_backward``) call
over the workload (forward recompute with every mini-batch's starting state
kept, then the reverse sweep), with seeded upstream gradients dZ and
final-state seeds. Its roofline is the fp32 FMA rate, since the kernels do
their contractions on the CUDA cores.
"""
from __future__ import annotations

import argparse
import functools
import json
import os
import statistics
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from test_weight_sequence_ttt_b300.inputs import WORKLOADS, make_cotangents, make_inputs  # noqa: E402

DEFAULT_WORKLOAD = "linear_b1h32_d64_t128k"
L2_FLUSH_BYTES = 256 << 20
CSRC = os.path.join(ROOT, "test_weight_sequence_ttt_b300", "csrc")
TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
# fp32 FFMA peak of one B300: 148 SMs x 128 FP32 lanes x 2 FLOP x 2.032 GHz (maximum SM clock)
FP32_PEAK_TFLOPS = 148 * 128 * 2 * 2.032e9 / 1e12
# dense tf32 over dense bf16 tensor throughput, nominal (1.1 / 2.25 PFLOP/s)
TF32_PER_BF16 = 1.1 / 2.25


# The source files each profiled kernel is built from (its .cu and the headers it includes).
KERNEL_SOURCES = {
    "linear_tc": ["ttt_linear_tc.cu", "tc_common.cuh", "ptx.cuh", "ttt_internal.h"],
    "mlp_tc": ["ttt_mlp_tc.cu", "tc_common.cuh", "ptx.cuh", "ttt_internal.h"],
    "linear_bwd": ["ttt_linear_bwd.cu", "ttt_internal.h"],
}


def _code_only(text: bytes) -> bytes:
    """The source without its C/C++ comments (so that a comment edit does not
    mark a measurement stale)."""
    import re
    t = re.sub(rb"/\*.*?\*/", b"", text, flags=re.S)
    return re.sub(rb"//[^\n]*", b"", t)


def sources_sha1(files=None) -> str:
    """sha1 over the code (comments removed) of CUDA sources of the library: the
    named files of csrc/, or all kernels and headers, and include/ttt.h."""
    import glob
    import hashlib
    h = hashlib.sha1()
    if files is None:
        paths = [f for f in sorted(glob.glob(os.path.join(CSRC, "*"))) if f.endswith((".cu", ".cuh", ".h"))]
    else:
        paths = [os.path.join(CSRC, f) for f in sorted(files)]
    for f in paths:
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode())
            h.update(_code_only(fh.read()))
    include = os.path.join(ROOT, "include", "ttt.h")
    with open(include, "rb") as fh:
        h.update(_code_only(fh.read()))
    return h.hexdigest()


def measured_traffic(workload: str, z_dtype: str, key: str = None):
    """DRAM bytes per launch of the workload's kernel from the last ncu capture
    (profiles/traffic.json), or None when the sources changed since."""
    try:
        with open(TRAFFIC) as f:
            j = json.load(f)
    except (OSError, ValueError):
        return None
    e = j.get(key or "%s/z_%s" % (workload, z_dtype))
    if not e or e.get("sources_sha1") != sources_sha1(e.get("sources")):
        return None
    return e.get("dram_bytes_per_launch")


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return dict(hbm_gbs=j["hbm_gbs"], bf16_tflops=j["bf16_tflops"],
                    bf16_tflops_sustained=j.get("bf16_tflops_sustained"), source="measured")
    return dict(hbm_gbs=6400.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0, source="fallback")


def algorithmic_cost(w, z_bytes: int = 4, out_rule: str = "prefix"):
    """Per-launch algorithmic bytes (Q/K/V in the io dtype, eta fp32, Z in its
    output dtype; the key output rule reads no Q) and dense-contraction FLOPs
    of the dual form."""
    es = 2 if w.io == "bf16" else 4
    per_tok_bytes = (2 if out_rule == "key" else 3) * w.d * es + 4 + w.d * z_bytes
    if w.variant == "linear":
        per_tok_flops = 6 * w.d * w.d + 4 * w.b * w.d
    else:
        h = w.hidden
        per_tok_flops = 14 * w.d * h + 4 * w.b * (w.d + h)
    return per_tok_bytes * w.tokens, per_tok_flops * w.tokens


def backward_cost(w):
    """Per-launch algorithmic bytes and FLOPs of ttt_linear_backward /
    ttt_mlp_backward.

    Bytes: K, V read by the forward sweep and Q, K, V, dZ by the reverse one
    (io dtype), eta twice, dQ, dK, dV, deta written fp32, plus every
    mini-batch's starting state (and for TTT-MLP its key-side activations)
    written once and read once. FLOPs, per
    mini-batch of b tokens, the contractions as executed: TTT-Linear
    10 b d^2 (forward recompute 2, reverse 8; 9 where the reverse sweep reuses
    the forward sweep's key side, d in {64, 128} and b = 16) + b^2 d (Q K^T) +
    5 b(b+1)/2 d (the causal b x b x d products); TTT-MLP 22 b h d (forward recompute 5,
    reverse 17: the reverse sweep reuses the forward sweep's key side) +
    b^2 (d + h) (the two Grams) + 5 b(b+1)/2 (d + h); times 2."""
    es = 2 if w.io == "bf16" else 4
    d, b = w.d, w.b
    saves = w.variant == "linear" and d in (64, 128) and b == 16  # keeps the key side: no V in the reverse
    per_tok = (2 * d * es) + ((3 if saves else 4) * d * es) + 2 * 4 + 3 * d * 4 + 4
    if w.variant == "linear":
        state = w.chains * (w.T // b) * (d * d + d) * 4 * 2
        if saves:
            state += w.tokens * (3 * d + 2) * 4 * 2
        flops_tok = 2 * ((9 if saves else 10) * d * d + b * d) + 5 * (b + 1) * d
    else:
        h = w.hidden
        state = (w.chains * (w.T // b) * (2 * h * d + h + d) + w.tokens * (2 * h + 3 * d + 2)) * 4 * 2
        flops_tok = 2 * (22 * h * d + b * (d + h)) + 5 * (b + 1) * (d + h)
    return per_tok * w.tokens + state, flops_tok * w.tokens


# ---------------------------------------------------------------- clocks (NVML, during the timed region)

class _NvmlCtypes:
    """The few NVML queries the sampler needs, through ctypes on the driver's
    libnvidia-ml.so.1 (read-only queries; present wherever the driver is)."""

    def __init__(self, bus_id: str):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        rc = self.lib.nvmlInit_v2()
        if rc != 0:
            raise RuntimeError("nvmlInit_v2 returned %d" % rc)
        self.h = ctypes.c_void_p()
        rc = self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus_id.encode(), ctypes.byref(self.h))
        if rc != 0:
            raise RuntimeError("nvmlDeviceGetHandleByPciBusId_v2(%s) returned %d" % (bus_id, rc))

    def clock(self, max_clock: bool = False) -> int:
        v = self.ct.c_uint()
        fn = self.lib.nvmlDeviceGetMaxClockInfo if max_clock else self.lib.nvmlDeviceGetClockInfo
        rc = fn(self.h, 1, self.ct.byref(v))  # 1 = NVML_CLOCK_SM
        if rc != 0:
            raise RuntimeError("clock query returned %d" % rc)
        return v.value

    def reasons(self) -> int:
        v = self.ct.c_ulonglong()
        rc = self.lib.nvmlDeviceGetCurrentClocksEventReasons(self.h, self.ct.byref(v))
        if rc != 0:
            raise RuntimeError("clocks event reasons query returned %d" % rc)
        return v.value


class ClockSampler:
    """Samples SM clock and clock-event (throttle) reasons of this process's GPU
    while the timed region runs: NVML (ctypes on the driver library, else the
    pynvml module) every 5 ms from a thread, else ``nvidia-smi -lms 50``. The
    sampler starts before the timed region; ``mark_start``/``mark_end`` bound
    it, and the summary keeps the samples inside it plus the last one before
    and the first one after (so a timed region shorter than the sampling period
    still has samples on both sides)."""
    REASONS = {
        0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
        0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
        0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting",
    }
    SMI_FIELDS = ["timestamp", "clocks.sm", "clocks.max.sm", "clocks_event_reasons.active"]

    def __init__(self, device_index: int, period_s: float = 0.005):
        self.period = period_s
        self.samples = []            # (time.perf_counter(), sm MHz, reason bits)
        self.max_mhz = None
        self.t_start = self.t_end = None
        self._stop = threading.Event()
        self._t = None
        self._proc = None
        self._q = None
        self.mode, self.error = None, None
        props = torch.cuda.get_device_properties(device_index)
        self.bus_id = "%08X:%02X:%02X.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id,
                                            props.pci_device_id)
        errs = []
        try:
            nv = _NvmlCtypes(self.bus_id)
            self._q = lambda: (nv.clock(), nv.reasons())
            self.max_mhz = nv.clock(max_clock=True)
            self.mode = "nvml-ctypes"
        except Exception as e:  # noqa: BLE001
            errs.append("nvml ctypes: %s" % e)
        if self.mode is None:
            try:
                import pynvml
                pynvml.nvmlInit()
                h = pynvml.nvmlDeviceGetHandleByPciBusId(self.bus_id.encode())
                self._q = lambda: (pynvml.nvmlDeviceGetClockInfo(h, pynvml.NVML_CLOCK_SM),
                                   pynvml.nvmlDeviceGetCurrentClocksEventReasons(h))
                self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(h, pynvml.NVML_CLOCK_SM)
                self.mode = "pynvml"
            except Exception as e:  # noqa: BLE001
                errs.append("pynvml: %s" % e)
        if self.mode is None:
            self.mode = "smi"
        self.error = "; ".join(errs) or None

    def _run_nvml(self):
        while not self._stop.is_set():
            try:
                mhz, bits = self._q()
                self.samples.append((time.perf_counter(), float(mhz), int(bits)))
            except Exception as e:  # noqa: BLE001
                self.error = "nvml sample: %s" % e
            time.sleep(self.period)

    def mark_start(self):
        self.t_start = time.perf_counter()

    def mark_end(self):
        self.t_end = time.perf_counter()
        if self.mode != "smi":
            time.sleep(3 * self.period)   # one sample after the region

    def __enter__(self):
        if self.mode != "smi":
            self._t = threading.Thread(target=self._run_nvml, daemon=True)
            self._t.start()
            time.sleep(3 * self.period)   # one sample before the region
        else:
            import subprocess
            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", "--id=" + self.bus_id, "--query-gpu=" + ",".join(self.SMI_FIELDS[1:]),
                     "--format=csv,noheader,nounits", "-lms", "50"],
                    stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
                time.sleep(0.3)           # nvidia-smi takes a moment to print its first line
            except Exception as e:  # noqa: BLE001
                self.error = (self.error or "") + "; smi: %s" % e
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._t:
            self._t.join()
        if self._proc:
            time.sleep(0.1)
            self._proc.terminate()
            out, err = self._proc.communicate(timeout=10)
            # nvidia-smi lines carry no host timestamp: keep them all (they span the region)
            for line in out.splitlines():
                f = [x.strip() for x in line.split(",")]
                try:
                    self.samples.append((None, float(f[0]), int(f[2], 16)))
                    self.max_mhz = float(f[1])
                except (ValueError, IndexError):
                    continue
            if not self.samples and err:
                self.error = (self.error or "") + "; smi: %s" % err.strip()[:200]

    def _window(self):
        if self.t_start is None or self.t_end is None or any(t is None for t, _, _ in self.samples):
            return list(self.samples)
        inside = [x for x in self.samples if self.t_start <= x[0] <= self.t_end]
        before = [x for x in self.samples if x[0] < self.t_start][-1:]
        after = [x for x in self.samples if x[0] > self.t_end][:1]
        return before + inside + after

    def summary(self):
        win = self._window()
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unavailable"], "samples": 0,
                    "error": self.error}
        bits = 0
        for _, _, b in win:
            bits |= b
        rs = [n for bit, n in sorted(self.REASONS.items()) if bits & bit]
        return {"sm_mhz": statistics.median(m for _, m, _ in win), "sm_max_mhz": self.max_mhz, "reasons": rs,
                "samples": len(win), "source": self.mode}


# ---------------------------------------------------------------- oracle timing

@functools.lru_cache(maxsize=4)
def _sample_inputs(w, n_chains: int, T: int, backward: bool = False):
    """fp64 numpy inputs (and, for the backward, upstream gradients) of the first
    ``n_chains`` chains and ``T`` tokens: drawn once per sample shape, so that a
    reference run of many steps spends its time in the oracle."""
    sel = list(range(n_chains))
    inp = make_inputs(w.with_(T=T), chains=sel)
    if backward:
        inp = dict(inp, **make_cotangents(w.with_(T=T), chains=sel))
    return {k: (v.detach().double().numpy() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def oracle_sample(w, n_chains: int, T: int, nthreads: int = 0, rule: str = "prefix"):
    """Run the fp64 oracle on the first ``n_chains`` chains, first ``T`` tokens.
    Returns (seconds, tokens processed, threads used)."""
    import oracle
    inp = _sample_inputs(w, n_chains, T)
    f = lambda t: t
    th = nthreads or oracle.max_threads()
    t0 = time.perf_counter()
    if w.variant == "linear":
        oracle.ttt_linear(f(inp["Q"]), f(inp["K"]), f(inp["V"]), f(inp["eta"]), f(inp["W0"]),
                          f(inp["c0"]), f(inp["ln_g"]), f(inp["ln_b"]), b=w.b, eps=w.eps,
                          nthreads=th, rule=rule, partial_tail=w.partial_tail)
    else:
        oracle.ttt_mlp(f(inp["Q"]), f(inp["K"]), f(inp["V"]), f(inp["eta"]), f(inp["W1"]), f(inp["c1"]),
                       f(inp["W2"]), f(inp["c2"]), f(inp["ln_g"]), f(inp["ln_b"]), b=w.b, eps=w.eps,
                       nthreads=th, rule=rule, partial_tail=w.partial_tail)
    dt = time.perf_counter() - t0
    return dt, n_chains * T, th


def _sample_shape(w, cpu_s: float, threads: int, calib=None):
    """Pick (chains, T') so one oracle call costs about ``cpu_s`` core-seconds
    spread over ``threads`` threads (calibrated on one short chain, single
    threaded; ``calib`` receives the single-thread tokens/s)."""
    Tc = max(w.b, min(w.T, (256 // w.b) * w.b or w.b))
    dt, toks, _ = oracle_sample(w, 1, Tc, nthreads=1)
    per_tok = dt / toks                                   # single-thread seconds per token-head
    if calib is not None:
        calib["single_thread_tokens_per_s"] = 1.0 / per_tok
        calib["single_thread_sample"] = "1 chain x %d tokens" % Tc
    tokens_budget = cpu_s / per_tok
    chains = int(min(w.chains, max(1, tokens_budget // w.T)))
    if chains >= threads and chains < w.chains:
        chains = chains // threads * threads   # whole rounds of the OpenMP threads over chains
    if chains >= threads or chains == w.chains:
        return chains, w.T
    chains = min(w.chains, threads)
    T = int(max(w.b, (tokens_budget / chains) // w.b * w.b))
    return chains, min(T, w.T)


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def oracle_backward_sample(w, n_chains: int, T: int):
    """Run the fp64 backward oracle (torch autograd through the primal token
    loop) on the first ``n_chains`` chains, first ``T`` tokens. Returns
    (seconds, tokens processed, threads used)."""
    from oracle.backward import ttt_linear_backward, ttt_mlp_backward
    inp = _sample_inputs(w, n_chains, T, backward=True)
    cot = inp
    f = lambda t: t
    t0 = time.perf_counter()
    if w.variant == "linear":
        ttt_linear_backward(f(inp["Q"]), f(inp["K"]), f(inp["V"]), f(inp["eta"]), f(inp["W0"]), f(inp["c0"]),
                            f(inp["ln_g"]), f(inp["ln_b"]), f(cot["dZ"]), f(cot["dW_n"]), f(cot["dc_n"]), b=w.b,
                            eps=w.eps)
    else:
        ttt_mlp_backward(*(f(inp[k]) for k in ("Q", "K", "V", "eta", "W1", "c1", "W2", "c2", "ln_g", "ln_b")),
                         f(cot["dZ"]), *(f(cot[k]) for k in ("dW1_n", "dc1_n", "dW2_n", "dc2_n")), b=w.b,
                         eps=w.eps)
    return time.perf_counter() - t0, n_chains * T, torch.get_num_threads()


def _backward_sample_shape(w, seconds: float):
    """(chains, T') for about ``seconds`` of backward-oracle time (calibrated on
    one short chain; the oracle is batched over chains, so chains cost less
    than linearly and this errs on the short side)."""
    Tc = max(w.b, min(w.T, (256 // w.b) * w.b or w.b))
    dt, toks, _ = oracle_backward_sample(w, 1, Tc)
    T = int(max(w.b, min(w.T, (seconds / (dt / Tc)) // w.b * w.b)))
    if T < w.T:
        return 1, T
    return int(min(w.chains, max(1, seconds / (dt / Tc * w.T)))), w.T


# ---------------------------------------------------------------- end to end

def pipelined_e2e(host_in: dict, dev_like: dict, out_like: dict, run, steps: int, warm: int = 2) -> float:
    """Seconds per step of ``steps`` end-to-end steps through the public API.

    Every step copies all of its inputs from pinned host memory to the device
    (``host_in``), runs ``run(dev_in, out, stream)`` and copies all of its
    results (``out``) back to pinned host memory, inside the timed region. As
    a user overlapping transfers with compute would, the steps are pipelined
    on three streams with two sets of buffers: step k's inputs go in while step
    k-1 computes, and step k-1's results come out while step k computes (PCIe
    carries both directions at once)."""
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    dev_in = [{k: torch.empty_like(v) for k, v in dev_like.items()} for _ in range(2)]
    outs = [{k: torch.empty_like(v) for k, v in out_like.items()} for _ in range(2)]
    host_out = [{k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in out_like.items()} for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    torch.cuda.synchronize()

    def step(k):
        j = k & 1
        if k >= 2:
            s_in.wait_event(ev_cmp[j])       # the compute that read dev_in[j] is done
        with torch.cuda.stream(s_in):
            for name, t in host_in.items():
                dev_in[j][name].copy_(t, non_blocking=True)
        ev_in[j].record(s_in)
        s_cmp.wait_event(ev_in[j])
        if k >= 2:
            s_cmp.wait_event(ev_out[j])      # outs[j] has been read back
        run(dev_in[j], outs[j], s_cmp)
        ev_cmp[j].record(s_cmp)
        s_out.wait_event(ev_cmp[j])
        with torch.cuda.stream(s_out):
            for name, t in host_out[j].items():
                t.copy_(outs[j][name], non_blocking=True)
        ev_out[j].record(s_out)

    for k in range(warm):
        step(k)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for k in range(steps):
        step(k)
    torch.cuda.synchronize()                  # every step's results are on the host
    return (time.perf_counter() - t0) / steps


# ---------------------------------------------------------------- GPU arm

def run_gpu_backward(args):
    """The --backward leg: ttt_linear_backward / ttt_mlp_backward over the whole workload."""
    import test_weight_sequence_ttt_b300 as ttt
    from test_weight_sequence_ttt_b300 import shard

    dist = shard.init()
    rank, world = shard.world()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    w = WORKLOADS[args.workload]
    if w.partial_tail or w.T % w.b:
        raise SystemExit("--backward needs a workload with T a multiple of mb")
    rank_chains = _rank_chains(dist, rank, world, w)
    wr = w.with_(seed=w.seed + 7919 * rank)
    inp = dict(make_inputs(wr), **make_cotangents(wr))
    eta_key = "eta_logit" if args.eta_gate else "eta"
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    stream = torch.cuda.current_stream()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    if w.variant == "linear":
        ws = torch.empty(ttt.linear_backward_workspace_bytes(w.B, w.H, w.T, w.d, w.b), dtype=torch.uint8,
                         device="cuda")
        seeds = ("dW_n", "dc_n")
        call = lambda o: ttt.ttt_linear_backward(dev["Q"], dev["K"], dev["V"], dev[eta_key], dev["W0"], dev["c0"],
                                                 dev["ln_g"], dev["ln_b"], dev["dZ"], mb=w.b, dW_n=dev["dW_n"],
                                                 dc_n=dev["dc_n"], eps=w.eps, out=o, workspace=ws, status=st,
                                                 stream=stream, eta_gate=args.eta_gate, eta_base=w.eta_base,
                                                 math=args.bwd_math)
    else:
        ws = torch.empty(ttt.mlp_backward_workspace_bytes(w.B, w.H, w.T, w.d, w.hidden, w.b), dtype=torch.uint8,
                         device="cuda")
        seeds = ("dW1_n", "dc1_n", "dW2_n", "dc2_n")
        call = lambda o: ttt.ttt_mlp_backward(*(dev[k] for k in ("Q", "K", "V")), dev[eta_key],
                                              *(dev[k] for k in ("W1", "c1", "W2", "c2", "ln_g", "ln_b", "dZ")),
                                              mb=w.b, eps=w.eps, out=o, workspace=ws, status=st, stream=stream,
                                              eta_gate=args.eta_gate, eta_base=w.eta_base,
                                              **{k: dev[k] for k in seeds})
    out = call({})
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    for _ in range(args.warmup):
        flush.fill_(1.0)
        call(out)
    torch.cuda.synchronize()
    if int(st.item()) != 0:
        raise RuntimeError("device status %d after warm-up" % int(st.item()))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sampler = ClockSampler(torch.cuda.current_device())
    shard.barrier(dist)
    torch.cuda.synchronize()
    with sampler:
        sampler.mark_start()
        wall0 = time.perf_counter()
        for e0, e1 in evs:
            flush.fill_(1.0)
            e0.record(stream)
            call(out)
            e1.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
        sampler.mark_end()
    shard.barrier(dist)
    times_ms = [a.elapsed_time(b) for a, b in evs]
    ms = statistics.mean(times_ms)
    ms_max = shard.max_over_ranks(dist, ms)
    if int(st.item()) != 0:
        raise RuntimeError("device status %d in timed region" % int(st.item()))

    # e2e: inputs and upstream gradients from pinned host memory, every gradient back to the host
    host_in = {k: inp[k].pin_memory() for k in ("Q", "K", "V", eta_key, "dZ") + seeds}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in out.values())
    e2e_steps = max(3, min(args.steps, 20))

    def run_e2e(di, o, strm):
        x = dict(dev, **di)
        if w.variant == "linear":
            ttt.ttt_linear_backward(x["Q"], x["K"], x["V"], x[eta_key], x["W0"], x["c0"], x["ln_g"], x["ln_b"],
                                    x["dZ"], mb=w.b, dW_n=x["dW_n"], dc_n=x["dc_n"], eps=w.eps, out=o,
                                    workspace=ws, status=st, stream=strm, eta_gate=args.eta_gate,
                                    eta_base=w.eta_base, math=args.bwd_math)
        else:
            ttt.ttt_mlp_backward(*(x[k] for k in ("Q", "K", "V")), x[eta_key],
                                 *(x[k] for k in ("W1", "c1", "W2", "c2", "ln_g", "ln_b", "dZ")), mb=w.b, eps=w.eps,
                                 out=o, workspace=ws, status=st, stream=strm, eta_gate=args.eta_gate,
                                 eta_base=w.eta_base, **{k: x[k] for k in seeds})

    shard.barrier(dist)
    e2e_s = pipelined_e2e(host_in, {k: dev[k] for k in host_in}, out, run_e2e, e2e_steps)
    e2e_s = shard.max_over_ranks(dist, e2e_s)
    tokens = shard.sum_over_ranks(dist, w.tokens)
    if rank != 0:
        return None
    bytes_launch, flops_launch = backward_cost(w)
    achieved = flops_launch / (ms / 1e3) / 1e12
    # TTT-Linear at d = 64 / 128, b = 16: the contractions run on the tensor cores with tf32
    # operands, split into hi + lo parts (three products each, two where one operand is a bf16
    # input) unless --bwd-math tf32; the fraction counts the algorithmic FLOPs once.
    tc = w.variant == "linear" and w.d in (64, 128) and w.b == 16
    split = tc and args.bwd_math == "fp32"
    if tc:
        pk = _peaks()
        peak, bound = pk["bf16_tflops"] * TF32_PER_BF16, "tensor"
        peak_src = "%s bf16 burst x %.3f (nominal dense tf32 / bf16, 1.1 / 2.25 PFLOP/s)" % (pk["source"],
                                                                                              TF32_PER_BF16)
    else:
        peak, bound = FP32_PEAK_TFLOPS, "alu"
        peak_src = "derived: 148 SMs x 128 FP32 lanes x 2 FLOP x 2.032 GHz"
    line = {
        "metric": "TTT-%s backward (outer-loop gradient) tokens/sec (B·T·H/s) on 1 B300"
                  % ("Linear" if w.variant == "linear" else "MLP"),
        "value": tokens / (ms_max / 1e3), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": ("tf32x3-mma/f32" if split else "tf32-mma/f32") if tc else "f32",
        "precision": "bf16 Q/K/V/dZ inputs; fp32 FFMA arithmetic, fp32 gradients",
        "data": "synthetic (seeded Gaussian Q/K/V/dZ, sigmoid-gated eta, N(0,0.02^2) W0)",
        "config": {"workload": w.name, "direction": "backward", "variant": "ttt-" + w.variant, "B": w.B,
                   "H": w.H, "T": w.T, "d": w.d, "mb": w.b, "hidden": w.hidden or None, "io": w.io,
                   "eta_gate": args.eta_gate,
                   "workspace_bytes": ws.numel(), "l2": "flushed between steps (256 MiB write)",
                   "parallelism": "dp%d" % world, "rank_chains": rank_chains},
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     "traffic": measured_traffic(w.name, "", key="%s/backward" % w.name) if not tc else None,
                     "peak_source": peak_src,
                     "algorithmic_bytes_per_launch": bytes_launch, "algorithmic_flops_per_launch": flops_launch},
        "e2e": {"value": tokens / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps,
        "clocks": sampler.summary(),
        "ms_per_step_min": min(times_ms), "ms_per_step_median": statistics.median(times_ms),
        "timed_wall_s": wall,
    }
    if world == 1 and not args.no_cpu_baseline:
        chains, Ts = _backward_sample_shape(w, args.cpu_budget_s / max(1, torch.get_num_threads()))
        dt, toks, th = oracle_backward_sample(w, chains, Ts)
        line["cpu_baseline"] = {"value": toks / dt, "unit": "tokens/s", "cores": th, "kind": "oracle",
                                "sample": "%d of %d chains x %d tokens (fp64 torch autograd through the "
                                          "primal token loop)" % (chains, w.chains, Ts), "seconds": dt}
    if split:
        line["precision"] = ("%s Q/K/V/dZ inputs; tensor-core products of fp32 operands split into tf32 hi + lo "
                             "parts (hi.hi + hi.lo + lo.hi, fp32 accumulation), fp32 LayerNorm rows and gradients"
                             % w.io)
    elif tc:
        line["precision"] = ("%s Q/K/V/dZ inputs; tensor-core products with tf32 operands and fp32 accumulation, "
                             "fp32 LayerNorm rows and gradients" % w.io)
    else:
        line["precision"] = "%s Q/K/V/dZ inputs; fp32 FFMA arithmetic, fp32 gradients" % w.io
    line["config"]["math"] = args.bwd_math
    return line


def run_gpu(args):
    import test_weight_sequence_ttt_b300 as ttt
    from test_weight_sequence_ttt_b300 import shard

    dist = shard.init()
    rank, world = shard.world()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    w = WORKLOADS[args.workload]
    ttt.linear_cluster_mode({"one_cta": 0, "auto": 1, "cluster": 2}[args.linear_form])
    ttt.mlp_cluster_mode({"one_cta": 0, "auto": 1, "cluster": 2}[args.mlp_form])
    # weak scaling: every rank runs its own full workload (independent chains)
    rank_chains = _rank_chains(dist, rank, world, w)
    inp = make_inputs(w.with_(seed=w.seed + 7919 * rank))
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    stream = torch.cuda.current_stream()
    B, H, T, d = dev["Q"].shape
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    zdt = torch.float32 if args.z_dtype == "f32" else torch.bfloat16
    out = {"Z": torch.empty(dev["Q"].shape, dtype=zdt, device="cuda")}

    rule = args.out_rule
    q_in = None if rule == "key" else dev["Q"]    # the key rule reads no queries
    eta_key = "eta_logit" if args.eta_gate else "eta"  # gate logits: the kernels apply the gate
    if w.variant == "linear":
        call = lambda o: ttt.ttt_linear_forward(q_in, dev["K"], dev["V"], dev[eta_key], dev["W0"], dev["c0"],
                                                dev["ln_g"], dev["ln_b"], mb=w.b, eps=w.eps, out=o,
                                                status=st, stream=stream, out_rule=rule,
                                                partial_tail=w.partial_tail, eta_gate=args.eta_gate,
                                                eta_base=w.eta_base)
        kind = ttt.linear_kernel_kind(ttt.BF16 if w.io == "bf16" else ttt.F32, w.d, w.b)
    else:
        call = lambda o: ttt.ttt_mlp_forward(q_in, dev["K"], dev["V"], dev[eta_key], dev["W1"], dev["c1"],
                                             dev["W2"], dev["c2"], dev["ln_g"], dev["ln_b"], mb=w.b, eps=w.eps,
                                             out=o, status=st, stream=stream, out_rule=rule,
                                             partial_tail=w.partial_tail, eta_gate=args.eta_gate,
                                             eta_base=w.eta_base)
        kind = ttt.mlp_kernel_kind(ttt.BF16 if w.io == "bf16" else ttt.F32, w.d, w.hidden, w.b)
    out = call(out)                       # allocates outputs once
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")

    for _ in range(args.warmup):
        flush.fill_(1.0)
        call(out)
    torch.cuda.synchronize()
    if int(st.item()) != 0:
        raise RuntimeError("device status %d after warm-up" % int(st.item()))

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sampler = ClockSampler(torch.cuda.current_device())
    shard.barrier(dist)
    torch.cuda.synchronize()
    with sampler:
        sampler.mark_start()
        wall0 = time.perf_counter()
        for e0, e1 in evs:
            flush.fill_(1.0)              # evict L2 (some workloads are smaller than it) -- outside the events
            e0.record(stream)
            call(out)
            e1.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
        sampler.mark_end()
    shard.barrier(dist)
    times_ms = [a.elapsed_time(b) for a, b in evs]
    ms = statistics.mean(times_ms)
    ms_max = shard.max_over_ranks(dist, ms)
    if int(st.item()) != 0:
        raise RuntimeError("device status %d in timed region" % int(st.item()))

    # ---- e2e: pinned host buffers through the C ABI, copies inside the timed region
    host_in = {k: inp[k].pin_memory() for k in (("K", "V", eta_key) if rule == "key" else ("Q", "K", "V", eta_key))}
    res = dict(out)      # every output of the call (Z, final W and c, loss, inner loss) is read back
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in res.values())
    e2e_steps = max(3, min(args.steps, 50))

    def run_e2e(di, o, strm):
        x = dict(dev, **di)
        qx = None if rule == "key" else x["Q"]
        if w.variant == "linear":
            ttt.ttt_linear_forward(qx, x["K"], x["V"], x[eta_key], x["W0"], x["c0"], x["ln_g"], x["ln_b"], mb=w.b,
                                   eps=w.eps, out=o, status=st, stream=strm, out_rule=rule,
                                   partial_tail=w.partial_tail, eta_gate=args.eta_gate, eta_base=w.eta_base)
        else:
            ttt.ttt_mlp_forward(qx, x["K"], x["V"], x[eta_key], x["W1"], x["c1"], x["W2"], x["c2"], x["ln_g"],
                                x["ln_b"], mb=w.b, eps=w.eps, out=o, status=st, stream=strm, out_rule=rule,
                                partial_tail=w.partial_tail, eta_gate=args.eta_gate, eta_base=w.eta_base)

    shard.barrier(dist)
    e2e_s = pipelined_e2e(host_in, {k: dev[k] for k in host_in}, res, run_e2e, e2e_steps)
    e2e_s = shard.max_over_ranks(dist, e2e_s)
    tokens = shard.sum_over_ranks(dist, w.tokens)  # every rank ran its own full workload (weak scaling)

    if rank != 0:
        return None
    peaks = _peaks()
    bytes_launch, flops_launch = algorithmic_cost(w, 4 if args.z_dtype == "f32" else 2, rule)
    value = tokens / (ms_max / 1e3)
    if w.variant == "linear":
        bound, achieved, peak, unit = "hbm", bytes_launch / (ms / 1e3) / 1e9, peaks["hbm_gbs"], "GB/s"
    else:
        bound, achieved, peak, unit = "tensor", flops_launch / (ms / 1e3) / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    t_roof = max(bytes_launch / (peaks["hbm_gbs"] * 1e9), flops_launch / (peaks["bf16_tflops"] * 1e12))
    line = {
        "metric": "TTT inner-loop tokens/sec (B·T·H/s) and % of roofline on 1 B300",
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_max,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16-mma/f32" if kind == 2 else "f32",
        "precision": "bf16 Q/K/V; fp16 tensor-core operands with fp32 accumulation; fp32 LayerNorm, "
                     "gradients and weight state" if kind == 2 else "fp32 FFMA",
        "data": "synthetic (seeded Gaussian Q/K/V, sigmoid-gated eta, N(0,0.02^2) W0)",
        "config": {"workload": w.name, "variant": "ttt-" + w.variant, "B": w.B, "H": w.H, "T": w.T, "d": w.d,
                   "mb": w.b, "hidden": w.hidden or None, "io": w.io, "z_dtype": args.z_dtype,
                   "out_rule": rule, "partial_tail": w.partial_tail, "eta_gate": args.eta_gate, "kernel_kind": kind,
                   "l2": "flushed between steps (256 MiB write)", "parallelism": "dp%d" % world,
                   "rank_chains": rank_chains, "linear_form": args.linear_form,
                   "mlp_form": args.mlp_form},
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak,
                     "traffic": measured_traffic(w.name, args.z_dtype) if rule == "prefix" else None,
                     "roofline_frac": t_roof / (ms / 1e3),
                     "peak_source": peaks["source"] + " (burst)",
                     "algorithmic_bytes_per_launch": bytes_launch, "algorithmic_flops_per_launch": flops_launch},
        "e2e": {"value": tokens / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps,
        "clocks": sampler.summary(),
        "ms_per_step_min": min(times_ms), "ms_per_step_median": statistics.median(times_ms),
        "timed_wall_s": wall,
    }
    if world == 1 and not args.no_cpu_baseline:
        threads = __import__("oracle").max_threads()
        calib = {}
        chains, Ts = _sample_shape(w, args.cpu_budget_s, threads, calib)
        oracle_sample(w, chains, Ts, nthreads=threads, rule=args.out_rule)       # warm-up call
        runs = [oracle_sample(w, chains, Ts, nthreads=threads, rule=args.out_rule) for _ in range(3)]
        dt = statistics.median(r[0] for r in runs)
        toks, th = runs[0][1], runs[0][2]
        line["cpu_baseline"] = {"value": toks / dt, "unit": "tokens/s", "cores": th, "kind": "oracle",
                                "sample": "%d of %d chains x %d tokens (fp64 primal token loop, C, OpenMP); "
                                          "median of 3 calls after one warm-up call" % (chains, w.chains, Ts),
                                "seconds": dt, "cpu_count": os.cpu_count(), "model": cpu_model(), **calib}
    return line


def _rank_chains(dist, rank: int, world: int, w):
    """Every rank's [start, stop) range of the job's chains. The job is ``world``
    workloads of ``w``'s shape (weak scaling); rank r owns the r-th block of
    w.chains chains, drawn from its own seed."""
    mine = list(shard_slice(rank, world, world * w.chains))
    if dist is None:
        return [mine]
    got = [None] * world
    dist.all_gather_object(got, mine)
    return got


def shard_slice(rank, world, n):
    from test_weight_sequence_ttt_b300 import shard
    return shard.chain_slice(rank, world, n)


def run_host_only(args):
    """The multi-process logic of the GPU arm on CPU (gloo): each rank's step is
    the fp64 oracle on a small slice of its own chains; barrier, max over ranks
    of the step time, sum of tokens, rank 0 prints the line."""
    from test_weight_sequence_ttt_b300 import shard
    dist = shard.init("gloo")
    rank, world = shard.world()
    w = WORKLOADS[args.workload]
    rank_chains = _rank_chains(dist, rank, world, w)
    wr = w.with_(seed=w.seed + 7919 * rank)
    n, Ts = min(2, w.chains), min(w.T, 2 * w.b)
    for _ in range(args.warmup):
        oracle_sample(wr, n, Ts, nthreads=1)
    shard.barrier(dist)
    secs = 0.0
    for _ in range(args.steps):
        dt, toks, _ = oracle_sample(wr, n, Ts, nthreads=1)
        secs += dt
    shard.barrier(dist)
    ms_max = shard.max_over_ranks(dist, 1e3 * secs / args.steps)
    tokens = shard.sum_over_ranks(dist, n * Ts)
    if rank != 0:
        return None
    return {"impl": "host-only", "metric": "TTT inner-loop tokens/sec (B·T·H/s) and % of roofline on 1 B300",
            "value": tokens / (ms_max / 1e3), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (same seeded generator)",
            "config": {"workload": w.name, "parallelism": "dp%d" % world, "rank_chains": rank_chains,
                       "sample": "%d chains x %d tokens per rank and step (CPU oracle stands in for the GPU)"
                                 % (n, Ts)}}


def _launch_ranks(args, argv):
    """Start ``args.gpus`` ranks of this script under torch.distributed.run
    (one process per GPU, rendezvous on 127.0.0.1) and return their exit code."""
    import socket
    import subprocess
    sk = socket.socket()
    sk.bind(("127.0.0.1", 0))
    port = sk.getsockname()[1]
    sk.close()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", str(args.gpus),
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *argv]
    return subprocess.call(cmd, cwd=ROOT)


# ---------------------------------------------------------------- reference arm: the oracle

def run_reference_backward(args):
    w = WORKLOADS[args.workload]
    per_step = max(0.2, args.ref_budget_s / max(1, args.steps + args.warmup))
    chains, Ts = _backward_sample_shape(w, per_step)
    for _ in range(args.warmup):
        oracle_backward_sample(w, chains, Ts)
    secs, toks, th = 0.0, 0, 1
    for _ in range(args.steps):
        dt, n, th = oracle_backward_sample(w, chains, Ts)
        secs += dt
        toks += n
    value = toks / secs
    return {
        "impl": "reference",
        "metric": "TTT-%s backward (outer-loop gradient) tokens/sec (B·T·H/s) on 1 B300"
                  % ("Linear" if w.variant == "linear" else "MLP"),
        "value": value, "unit": "tokens/s", "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (same seeded generator)",
        "config": {"workload": w.name, "direction": "backward", "variant": "ttt-" + w.variant, "B": w.B,
                   "H": w.H, "T": w.T, "d": w.d, "mb": w.b, "hidden": w.hidden or None},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": th, "kind": "oracle",
                         "sample": "%d of %d chains x %d tokens per step" % (chains, w.chains, Ts)},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    if args.backward:
        return run_reference_backward(args)
    import oracle
    w = WORKLOADS[args.workload]
    threads = oracle.max_threads()
    # at least 0.05 s of oracle work per step, so fixed per-call costs (thread
    # start, state set-up) stay small next to it
    per_step_wall = max(0.05, args.ref_budget_s / max(1, args.steps + args.warmup))
    chains, Ts = _sample_shape(w, per_step_wall * threads, threads)
    for _ in range(args.warmup):
        oracle_sample(w, chains, Ts, nthreads=threads, rule=args.out_rule)
    secs, toks = 0.0, 0
    for _ in range(args.steps):
        dt, n, _ = oracle_sample(w, chains, Ts, nthreads=threads, rule=args.out_rule)
        secs += dt
        toks += n
    value = toks / secs
    return {
        "impl": "reference",
        "metric": "TTT inner-loop tokens/sec (B·T·H/s) and % of roofline on 1 B300",
        "value": value, "unit": "tokens/s", "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (same seeded generator)",
        "config": {"workload": w.name, "variant": "ttt-" + w.variant, "B": w.B, "H": w.H, "T": w.T, "d": w.d,
                   "mb": w.b, "hidden": w.hidden or None, "out_rule": args.out_rule},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": "%d of %d chains x %d tokens per step" % (chains, w.chains, Ts),
                         "cpu_count": os.cpu_count(), "model": cpu_model()},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--z-dtype", default="bf16", choices=["f32", "bf16"],
                    help="element type of Z (bf16 = the I/O type of the workloads)")
    ap.add_argument("--cpu-budget-s", type=float, default=20.0, help="core-seconds of the oracle sample")
    ap.add_argument("--ref-budget-s", type=float, default=60.0,
                    help="seconds of oracle time the reference arm aims for over all its steps")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eta-gate", action="store_true",
                    help="pass the learning-rate gate logits; the kernels apply eta_base * sigmoid()")
    ap.add_argument("--T", type=int, default=0,
                    help="tokens per chain instead of the workload's (a small case of the same kernel, "
                         "for profiling; the line's config says so)")
    ap.add_argument("--backward", action="store_true",
                    help="time ttt_linear_backward (gradients through the inner loop) instead of the forward")
    ap.add_argument("--bwd-math", default="fp32", choices=["fp32", "tf32"],
                    help="TTT-Linear backward: fp32 FFMA products, or tf32 tensor-core products (d=64, b=16)")
    ap.add_argument("--linear-form", default="one_cta", choices=["one_cta", "cluster", "auto"],
                    help="d=64, b=16 TTT-Linear kernel form: one CTA per chain (default), a two-CTA cluster per "
                         "chain, or the cluster when 2*B*H <= SMs (ttt_linear_cluster_mode 0 / 2 / 1)")
    ap.add_argument("--mlp-form", default="auto", choices=["one_cta", "cluster", "auto"],
                    help="tensor-core TTT-MLP kernel form: one CTA per chain, a two-CTA cluster per chain with the "
                         "hidden units split, or the cluster when 2*B*H <= SMs (default; ttt_mlp_cluster_mode 0 / 2 / 1)")
    ap.add_argument("--host-only", action="store_true",
                    help="run the multi-rank logic on CPU (gloo) with the oracle standing in for the GPU step")
    ap.add_argument("--out-rule", default="prefix", choices=["prefix", "anchor", "key"],
                    help="output rule: z_t = f(q_t; W_t) (prefix), f(q_t; W_{i-1}) (anchor), f(k_t; W_{i-1}) (key)")
    raw = list(sys.argv[1:] if argv is None else argv)
    args = ap.parse_args(raw)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    if "WORLD_SIZE" in os.environ:
        if int(os.environ["WORLD_SIZE"]) != args.gpus:
            ap.error("--gpus %d but WORLD_SIZE=%s" % (args.gpus, os.environ["WORLD_SIZE"]))
    elif args.gpus > 1:
        raise SystemExit(_launch_ranks(args, raw))
    if args.T:
        name = "%s_T%d" % (args.workload, args.T)
        WORKLOADS[name] = WORKLOADS[args.workload].with_(name=name, T=args.T)
        args.workload = name
    if args.backward and args.out_rule != "prefix":
        ap.error("--backward supports the prefix output rule only")
    if args.impl == "reference":
        line = run_reference(args)
    elif args.host_only:
        line = run_host_only(args)
    else:
        line = run_gpu_backward(args) if args.backward else run_gpu(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
