"""The multi-process pieces of bench.py on the CPU: two gloo ranks on 127.0.0.1.

bench.py runs one replica per GPU (there is no exchange step on this path); what the ranks share
is the timing rule -- a barrier before the timed region and the maximum of the ranks' times -- and
which rank prints.  These run here without a GPU.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench._dist()
        assert (ws, r, local) == (world, rank, rank)
        dist.barrier()
        # rank-dependent "times": everyone must see the slowest
        got = bench.max_over_ranks(1.5 + rank * 2.25, torch.device("cpu"))
        out.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(out.get(timeout=10) for _ in range(2))
    assert res == {0: 3.75, 1: 3.75}


def test_max_over_ranks_without_a_group():
    import torch
    import bench
    assert bench.max_over_ranks(2.5, torch.device("cpu")) == 2.5


def test_reference_arm_other_ranks_exit_silently():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
