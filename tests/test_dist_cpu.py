"""The multi-process path of bench.py on CPU: two ranks over gloo run the
same setup, barrier and max-over-ranks helpers the GPU runs use over NCCL
(one process per GPU, replicas with no data-path collective), and the
reference arm does its work on rank 0 only."""
import argparse
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _rank(rank, port, results):
    os.environ.update(WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    world, r, _ = bench.dist_setup()
    bench.barrier(world)
    slowest = bench.max_over_ranks(10.0 * (r + 1), world)  # per-rank "times" 10 and 20
    results.put((r, world, dist.get_backend(), slowest))
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_ranks_over_gloo():
    ctx = mp.get_context("spawn")
    results = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    assert [p.exitcode for p in procs] == [0, 0]
    got = sorted(results.get(timeout=10) for _ in range(2))
    assert got == [(0, 2, "gloo", 20.0), (1, 2, "gloo", 20.0)]


def test_reference_arm_works_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    # rank 1 returns at once: no inputs are built, nothing is timed or printed
    assert bench.run_reference(argparse.Namespace(steps=1, warmup=0)) is None
