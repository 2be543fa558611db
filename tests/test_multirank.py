"""The N > 1 path on CPU with gloo: one independent episode per rank (weak scaling), no
collective on the data path, a max over ranks of the step time.  Each rank checks its
own episode's plan layout against the oracle (plans are integer work the oracle derives
on the CPU), so the test needs no GPU."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import synth


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    import oracle
    oracle.build()
    seed = bench.rank_seed(0, rank)
    ep = synth.random_dag(seed, page_size=16, max_segments=10, max_len=60)
    orc = oracle.Oracle(16, 512, 1, 64)
    orc.replay(ep)
    pl = orc.pack(ep.roots, 32)
    units = pl.pairs                       # this rank's useful work
    t_local = 1.0 + rank                   # stand-in step time of this rank
    t = bench.max_over_ranks(t_local, dist)
    tot = torch.tensor([float(units)])
    dist.all_reduce(tot)                   # test-side check only: the sum of all ranks' work
    out[rank] = (seed, units, t, float(tot.item()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_independent_episodes():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    port = _free_port()
    mp.get_context("spawn")
    procs = [mp.get_context("spawn").Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    seeds = [out[r][0] for r in range(world)]
    assert len(set(seeds)) == world                       # each rank its own episode
    assert all(out[r][2] == 1.0 + (world - 1) for r in range(world))   # max over ranks
    assert out[0][3] == out[0][1] + out[1][1]
