"""The replica (weak-scaling) aggregation of bench.py on two gloo ranks -- CPU only.

The path has no exchange step: N GPUs run N independent replicas.  What the ranks share
is the job's clock (the slowest replica) and the summed throughput."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [12.5, 17.25][rank]
        slowest = bench.max_over_ranks(ms)
        dist.barrier()
        q.put((rank, bench.dist_info(), slowest, bench.job_throughput(100.0, world, slowest * 1e-3)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (r, w, lr), slowest, thr in out:
        assert (r, w, lr) == (rank, 2, rank)
        assert slowest == 17.25
        assert thr == pytest.approx(100.0 * 2 / 17.25e-3)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_throughput(10.0, 1, 2.0) == 5.0
