"""The N > 1 host logic of bench.py on CPU: two gloo ranks, each timing its own
replica, agree on the barrier and on the maximum over ranks; under torchrun
the reference arm runs on rank 0 alone."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    ctx = bench.dist_setup(world)
    ctx["dist"].init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.dist_barrier(ctx)
        got = bench.dist_max(ctx, 10.0 + rank * 5.0)   # rank r "measured" 10 + 5r ms
        q.put((rank, ctx["world"], got))
    finally:
        ctx["dist"].destroy_process_group()


def test_two_gloo_ranks_take_the_max():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(world))
    assert res == [(0, 2, 15.0), (1, 2, 15.0)]


def test_reference_arm_runs_on_rank_zero_only():
    """A rank other than 0 exits 0 at once without work or output."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1",
               MASTER_PORT=str(_free_port()))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""
