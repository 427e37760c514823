"""Child process of tests/test_failure_detection.py (GPU).

Loads the library built with the fault hook, makes the loader drop one
super-step's tiles so every consumer's bounded wait runs out, and reports the
device status of the TTT-Linear and TTT-MLP calls, how long they took, and
whether a normal call afterwards (hook off) in the same context is correct.
Prints one JSON line.
"""
import ctypes
import json
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import torch  # noqa: E402

import test_weight_sequence_ttt_b300 as ttt  # noqa: E402
from test_weight_sequence_ttt_b300 import build as B  # noqa: E402
from test_weight_sequence_ttt_b300.inputs import WORKLOADS, make_inputs  # noqa: E402

from _util import dev, oracle_linear, rel_err, to_np  # noqa: E402

ttt.lib_path = B.build_faults()
L = ttt.lib()
L.ttt_debug_drop_load.restype = ctypes.c_int
L.ttt_debug_drop_load.argtypes = [ctypes.c_int32]
res = {"hook": L.ttt_debug_drop_load(2)}

lin = make_inputs(WORKLOADS["linear_b8h12_d64_t2k"].with_(B=2, H=2, T=96, seed=501))
mlp = make_inputs(WORKLOADS["mlp_b4h12_d64_t8k"].with_(B=1, H=2, T=96, seed=502))


def run_linear(inp):
    d = dev(inp)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    o = ttt.ttt_linear_forward(d["Q"], d["K"], d["V"], d["eta"], d["W0"], d["c0"], d["ln_g"], d["ln_b"],
                               mb=inp["b"], eps=inp["eps"], status=st)
    torch.cuda.synchronize()
    return o, int(st.item()), time.perf_counter() - t0


def run_mlp(inp):
    d = dev(inp)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    o = ttt.ttt_mlp_forward(d["Q"], d["K"], d["V"], d["eta"], d["W1"], d["c1"], d["W2"], d["c2"], d["ln_g"],
                            d["ln_b"], mb=inp["b"], eps=inp["eps"], status=st)
    torch.cuda.synchronize()
    return o, int(st.item()), time.perf_counter() - t0


_, res["linear_status"], res["linear_s"] = run_linear(lin)
ttt.mlp_cluster_mode(0)   # one CTA per chain
_, res["mlp_status"], res["mlp_s"] = run_mlp(mlp)
ttt.mlp_cluster_mode(2)   # two-CTA clusters: both CTAs time out, their exchanges stay in step
_, res["mlp_cluster_status"], res["mlp_cluster_s"] = run_mlp(mlp)
ttt.mlp_cluster_mode(1)
res["hook_off"] = L.ttt_debug_drop_load(-1)
o, res["after_status"], _ = run_linear(lin)
res["after_err"] = rel_err(to_np(o["Z"]), oracle_linear(lin)["Z"])
print(json.dumps(res))
