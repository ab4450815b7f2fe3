"""Multi-GPU is replicas only: sequences shard across ranks with no collective
on the decode path.  bench.py's cross-rank reduction (max of the ranks'
times, sum of their tokens) is checked with two gloo ranks on the CPU.
"""

import os

import torch.multiprocessing as mp


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms, toks = bench.aggregate(10.0 + rank, 100.0 * (rank + 1), world, device="cpu")
    out[rank] = (ms, toks)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation():
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == (11.0, 300.0)
    assert out[1] == (11.0, 300.0)


def test_single_rank_is_identity():
    import bench
    assert bench.aggregate(5.0, 7.0, 1) == (5.0, 7.0)
