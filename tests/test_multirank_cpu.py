"""The N>1 path of bench.py on CPU: two gloo ranks (127.0.0.1) reduce their
step times with max and their token counts with sum, the way the benchmark
does before rank 0 prints the whole-job throughput.  Replicas only: no data
path collective exists in the decode itself."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    t_max = bench.max_over_ranks(10.0 + rank, w, "cpu")
    tok = bench.sum_over_ranks(1000.0 * (rank + 1), w, "cpu")
    bench.barrier(w)
    q.put((rank, t_max, tok))
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_like_the_benchmark():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert res == [(0, 11.0, 3000.0), (1, 11.0, 3000.0)]
