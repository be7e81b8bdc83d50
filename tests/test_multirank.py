"""The multi-rank path of bench.py on CPU: two `gloo` ranks (world size 2).

Every rank of a GPU run is an independent replica (the problem splits by
batch and head with no exchange), so the only cross-rank steps are the timing
barrier and the maximum over ranks; the reference arm runs on rank 0 alone.
"""
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


def _worker(rank, port, out):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=2)
    try:
        dist.barrier()
        got = bench.max_over_ranks(dist, [1.0 + rank, 5.0 - rank, 0.25], "cpu")
        out[rank] = got
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(port, out), nprocs=2, join=True)
        assert out[0] == out[1] == [2.0, 5.0, 0.25]


def test_single_process_returns_the_values():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, [3, 4.5], "cpu") == [3.0, 4.5]


def test_reference_arm_prints_only_on_rank_zero():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "1", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip() == ""
