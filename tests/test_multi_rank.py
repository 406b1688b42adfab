"""The N>1 host path of bench.py on CPU: two gloo ranks (one process each, as
torchrun starts them). Every rank runs its own replica of the workload; the
timed region is bracketed by barriers and the job time is the maximum over the
ranks (``bench.max_over_ranks``); only rank 0 prints. No GPU is used."""
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        dist.barrier()
        got = bench.max_over_ranks(times[rank], world, torch.device("cpu"))
        dist.barrier()
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def _run(world, times):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return out


def test_job_time_is_the_slowest_rank_on_every_rank():
    assert _run(2, [3.5, 7.25]) == [(0, 7.25), (1, 7.25)]
    assert _run(2, [9.0, 1.0]) == [(0, 9.0), (1, 9.0)]


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(4.0, 1, torch.device("cpu")) == 4.0


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
