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


def _bench_run(args, env_extra):
    import subprocess
    env = dict(os.environ)
    env.pop("WORLD_SIZE", None)
    env.update(env_extra)
    env["CUDA_VISIBLE_DEVICES"] = ""          # no GPU: the refusal must come first
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, env=env,
                          capture_output=True, text=True, timeout=300)


def test_bench_refuses_a_world_size_other_than_gpus():
    r = _bench_run(["--gpus", "2", "--steps", "1", "--warmup", "1"], {"WORLD_SIZE": "3"})
    assert r.returncode != 0
    assert "WORLD_SIZE=3" in r.stderr
    assert '"n_gpus"' not in r.stdout


def test_bench_with_more_gpus_than_visible_never_prints_a_one_gpu_line():
    r = _bench_run(["--gpus", "2", "--steps", "1", "--warmup", "1"], {})
    assert r.returncode != 0
    assert "CUDA device" in r.stderr
    assert '"n_gpus"' not in r.stdout
