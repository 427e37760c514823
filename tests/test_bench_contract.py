"""Host-side checks of bench.py (no GPU): the reference arm's JSON line and the
algorithmic cost models the roofline divides by."""
import json
import os
import subprocess
import sys

import bench
from test_weight_sequence_ttt_b300.inputs import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                         timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    return json.loads(out.stdout.strip().splitlines()[-1])


def test_reference_arm_line():
    j = _run("--impl", "reference", "--steps", "1", "--warmup", "3", "--ref-budget-s", "2")
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in j, k
    assert j["impl"] == "reference" and j["value"] > 0 and j["unit"] == "tokens/s"
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["cores"] >= 1
    assert j["e2e"]["h2d_bytes_per_step"] == 0 and j["config"]["workload"] == bench.DEFAULT_WORKLOAD


def test_reference_arm_backward_line():
    j = _run("--impl", "reference", "--backward", "--steps", "1", "--warmup", "3", "--ref-budget-s", "2",
             "--workload", "linear_b8h12_d64_t2k", "--T", "64")
    assert j["config"]["direction"] == "backward" and j["value"] > 0


def test_cost_models():
    w = WORKLOADS["linear_b8h12_d64_t2k"]
    nbytes, flops = bench.algorithmic_cost(w, 2)
    assert nbytes == (3 * 64 * 2 + 4 + 64 * 2) * w.tokens          # 516 B per token-head
    assert flops == (6 * 64 * 64 + 4 * 16 * 64) * w.tokens          # 28 672 FLOP per token-head
    nb_key, _ = bench.algorithmic_cost(w, 2, "key")
    assert nb_key == nbytes - 64 * 2 * w.tokens                     # the key rule reads no queries
    bb, bf = bench.backward_cost(w)
    assert bf == (2 * (9 * 64 * 64 + 16 * 64) + 5 * 17 * 64) * w.tokens    # 81 216 FLOP per token-head
    assert bb == 1420 * w.tokens + w.chains * (2048 // 16) * (64 * 64 + 64) * 8 + w.tokens * 194 * 8
    m = WORKLOADS["mlp_b4h12_d64_t8k"]
    _, mf = bench.backward_cost(m)
    assert mf == (2 * (22 * 256 * 64 + 16 * (64 + 256)) + 5 * 17 * (64 + 256)) * m.tokens  # 758 336
    assert abs(bench.FP32_PEAK_TFLOPS - 148 * 128 * 2 * 2.032e-3) < 1e-9   # TFLOP/s


def test_two_ranks_host_only():
    """``--gpus 2`` without a torchrun environment starts the two ranks itself;
    rank 0 alone prints one line, for the whole job, and the ranks' chains are
    disjoint blocks that cover the job."""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--host-only",
                          "--steps", "2", "--warmup", "3", "--workload", "linear_b8h12_d64_t2k"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    j = json.loads(lines[0])
    assert j["n_gpus"] == 2 and j["scaling"] == "weak" and j["value"] > 0
    spans = j["config"]["rank_chains"]
    n = WORKLOADS["linear_b8h12_d64_t2k"].chains
    assert spans == [[0, n], [n, 2 * n]]
