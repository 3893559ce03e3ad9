"""The multi-rank (torchrun) path of the benchmark, on CPU with gloo.

Ranks decode independent sequences (weak scaling, no collective on the data
path); the only exchange is the max-over-ranks timing.  Two gloo ranks run the
oracle on their own seeded sequences and check that (a) the rank seeds give
different inputs, (b) the timing reduction returns the slowest rank's time on
every rank.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        from rs_decode_gb300 import synth
        w = synth.WORKLOADS["tiny"].with_(B=2)
        params = synth.layer_params(w)
        d = synth.step_inputs(w, 0, seed=bench.rank_seed(rank))
        y = oracle.Model("mamba2", synth.initial_state(w), params).step(d)
        fake_ms = 10.0 * (rank + 1)
        out[rank] = (bench.max_over_ranks(fake_ms), float(np.abs(y).sum()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0][0] == out[1][0] == 20.0     # slowest rank's time everywhere
    assert out[0][1] != out[1][1]             # independent sequences per rank


def test_single_process_max_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
