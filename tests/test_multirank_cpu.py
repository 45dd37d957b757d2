"""The N > 1 path of bench.py on CPU: two gloo ranks take the element-wise maximum of their
timings (the slowest replica sets the job time), and the reference arm does its work on rank 0
only (other ranks exit without output)."""
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


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        vals = [1.0 + rank, 10.0 - rank, 5.0, 0.5 * rank]
        out[rank] = bench.max_over_ranks(vals, torch.device("cpu"), world)
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    world = 2
    with mp.get_context("spawn").Manager() as m:    # no fork of this multi-threaded process
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        assert res[r] == [2.0, 10.0, 5.0, 0.5]


def test_reference_arm_nonzero_rank_is_silent():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "1"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
