"""Multi-process placement logic on CPU (gloo, world size 2).

Every chain is independent, so ranks split the chains with no data-path
exchange; these tests check the split and the host-side collectives that the
benchmark uses (max of step times, sum of tokens), and that the oracle run
rank by rank over the shards reassembles the single-process result.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from test_weight_sequence_ttt_b300 import shard
from test_weight_sequence_ttt_b300.inputs import WORKLOADS, make_inputs


@pytest.mark.parametrize("n,world", [(96, 2), (7, 3), (2, 4), (0, 2), (148, 8)])
def test_chain_slices_partition(n, world):
    spans = [shard.chain_slice(r, world, n) for r in range(world)]
    assert spans[0][0] == 0 and spans[-1][1] == n
    for (a, b), (c, d) in zip(spans, spans[1:]):
        assert b == c
    sizes = [b - a for a, b in spans]
    assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard.chain_slice(world, world, n)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _oracle_z(w, chains):
    import oracle
    inp = make_inputs(w, chains=chains)
    f = lambda t: t.double().numpy()
    out = oracle.ttt_linear(f(inp["Q"]), f(inp["K"]), f(inp["V"]), f(inp["eta"]), f(inp["W0"]), f(inp["c0"]),
                            f(inp["ln_g"]), f(inp["ln_b"]), b=w.b, eps=w.eps, nthreads=1)
    return out["Z"].reshape(len(chains), w.T, w.d)


def _worker(rank, world, port, wdict, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    from test_weight_sequence_ttt_b300.inputs import Workload
    dist = shard.init("gloo")
    try:
        w = Workload(**wdict)
        a, b = shard.chain_slice(rank, world, w.chains)
        sel = list(range(a, b))
        z = _oracle_z(w, sel)
        mx = shard.max_over_ranks(dist, 1.0 + rank)  # stand-in step times: the slowest rank decides
        tot = shard.sum_over_ranks(dist, float(len(sel) * w.T))
        shard.barrier(dist)
        q.put((rank, sel, z, mx, tot))
    finally:
        dist.destroy_process_group()


def test_two_rank_shards_reassemble_oracle():
    import dataclasses
    w = WORKLOADS["linear_b8h12_d64_t2k"].with_(B=1, H=5, T=32, d=16)
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, dataclasses.asdict(w), q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=120) for _ in procs), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert all(r[3] == float(world) for r in res)            # max over ranks
    assert all(r[4] == float(w.chains * w.T) for r in res)   # sum over ranks
    assert [c for r in res for c in r[1]] == list(range(w.chains))
    got = np.concatenate([r[2] for r in res], 0)
    np.testing.assert_array_equal(got, _oracle_z(w, list(range(w.chains))))
