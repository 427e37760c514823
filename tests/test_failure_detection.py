"""Failure detection on the GPU without a GPU fault.

Every wait of the tensor-core kernels is bounded (2 s); when one runs out the
chain records TTT_ERR_TIMEOUT in the caller's status word and every warp keeps
going in step (no early exit) until the kernel ends, so the context stays
usable. The library built with the fault hook makes the loader drop one
super-step's tiles (a barrier that nothing completes); the test checks the
status, that the call returned, and that a normal call afterwards in the same
process is correct. No trap, assert, bad address or endless loop is used.
"""
import ctypes
import json
import os
import subprocess
import sys

import pytest

import test_weight_sequence_ttt_b300 as ttt

HERE = os.path.dirname(os.path.abspath(__file__))
TIMEOUT = 7  # TTT_ERR_TIMEOUT


def test_product_library_has_no_hook():
    f = ttt.lib().ttt_debug_drop_load
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int32]
    assert f(3) == -1


@pytest.mark.gpu
def test_dropped_stage_reports_timeout_and_context_survives():
    r = subprocess.run([sys.executable, os.path.join(HERE, "_fault_child.py")], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["hook"] == 0 and res["hook_off"] == 0, res
    assert res["linear_status"] == TIMEOUT, res
    assert res["mlp_status"] == TIMEOUT and res["mlp_cluster_status"] == TIMEOUT, res
    assert max(res["linear_s"], res["mlp_s"], res["mlp_cluster_s"]) < 30, res   # bounded waits: the calls returned
    assert res["after_status"] == 0 and res["after_err"] <= 2e-2, res
