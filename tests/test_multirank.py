"""Host-side logic of the multi-process benchmark path, world size 2 on gloo
(CPU): every rank times its own copy of the workload (weak scaling, no
collective on the data path); the reported time is the max over ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    ws, r, local = bench._dist()
    assert (ws, r, local) == (world, rank, rank)
    dist = bench._init_dist(ws, "gloo")
    t = bench.reduce_max(10.0 + rank, ws)      # rank 1 is slower
    out[rank] = t
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_max_over_ranks_world_size_2():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert dict(out) == {0: 11.0, 1: 11.0}
