"""The N > 1 host logic of bench.py on CPU with the gloo backend, two ranks:
the timed region takes the slowest rank's time and the value counts every
rank's replica (weak scaling, no data-path collective)."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from paged_kv_attention_05_gb300 import workloads as W
    t = bench.max_over_ranks(1.0 + rank, dist, "cpu")       # rank 1 is slower
    spec = W.spec("mha_decode")
    v = bench.whole_job_value(bench.metric_work(spec), world, t)
    dist.barrier()
    q.put((rank, t, v))
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_sum_the_work():
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
    sys.path.insert(0, ROOT)
    import bench
    from paged_kv_attention_05_gb300 import workloads as W
    work = bench.metric_work(W.spec("mha_decode"))
    for rank, t, v in res:
        assert t == 2.0
        assert v == pytest.approx(2 * work / 2.0)
