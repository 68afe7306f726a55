"""The multi-rank path of bench.py on CPU: world-size-2 gloo process groups (no GPU)."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r took (1 + r) seconds for (100 * (r + 1)) bytes
    t, b = bench.whole_job(1.0 + rank, 100.0 * (rank + 1), torch.device("cpu"))
    q.put((rank, t, b))
    dist.barrier()
    dist.destroy_process_group()


def test_whole_job_takes_the_slowest_rank_and_all_bytes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, t, b in res:
        assert t == 2.0 and b == 300.0


def test_whole_job_single_process_is_a_pass_through():
    import torch
    sys.path.insert(0, ROOT)
    import bench
    assert bench.whole_job(1.5, 10.0, torch.device("cpu")) == (1.5, 10.0)


def test_reference_arm_prints_only_on_rank_zero():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "1"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
