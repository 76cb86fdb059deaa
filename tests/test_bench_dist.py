"""The multi-replica path of bench.py on CPU: two gloo ranks, max-over-ranks timing
and whole-job throughput (N independent replicas, no data-path collective)."""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    secs = [1.5, 2.0][rank]
    mx = bench.max_over_ranks(secs)
    value = bench.whole_job_throughput(10.0, world, mx)
    q.put((rank, mx, value))
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, value in res:
        assert mx == 2.0
        assert value == 10.0 * 2 / 2.0


def test_single_process_identity():
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.whole_job_throughput(8.0, 1, 2.0) == 4.0
