"""The multi-rank host logic of bench.py on CPU: two gloo ranks, the timing
reductions (max and sum over ranks) and a distinct batch per rank."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    from workloads import decode_config
    d = bench.Dist()
    d.init(torch, backend="gloo")
    d.barrier(torch)
    mx = d.max(torch, 1.5 + rank)
    sm = d.sum(torch, 10.0 * (rank + 1))
    case = decode_config(2, scale_down=32, seed_offset=d.rank)
    out[rank] = (mx, sm, int(case.cache_seqlens.sum()))
    d.close()


def test_two_gloo_ranks():
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 2.5          # max over ranks
    assert res[0][1] == res[1][1] == 30.0         # sum over ranks
    assert res[0][2] != res[1][2]                 # each rank has its own batch


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    assert d.world == int(os.environ.get("WORLD_SIZE", "1"))
    if d.world == 1:
        d.init(torch, backend="gloo")
        assert d.max(torch, 3.0) == 3.0 and d.sum(torch, 3.0) == 3.0
