"""The multi-GPU form of the path is independent replicas (decode batches do
not interact; expert-parallel exchange is out of scope). These CPU tests run
the bench's cross-rank reduction and its rank-0-only reporting with
world_size 2 over gloo."""

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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    # rank 0 streamed 3 GB in 2 ms, rank 1 streamed 5 GB in 4 ms
    b, ms, gbs = bench.aggregate([3e9, 5e9][rank], [2.0, 4.0][rank], dist, "cpu")
    q.put((rank, b, ms, gbs))
    dist.destroy_process_group()


def test_aggregate_sums_bytes_over_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(2))
    for rank, b, ms, gbs in res:
        assert b == 8e9 and ms == 4.0
        assert abs(gbs - 8e9 / 4e-3 / 1e9) < 1e-9


def test_single_process_aggregate_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate(1e9, 1.0) == (1e9, 1.0, 1000.0)


def test_reference_arm_only_rank0_prints():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                          "--steps", "1"], env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0
    assert out.stdout.strip() == ""
