"""Multi-process host logic of bench.py on CPU (gloo, world size 2): the job
time is the slowest rank's, the job's value counts every rank's replica, and
the CPU reference arm runs on rank 0 only."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(10.0 + rank)            # rank 1 is slower
        units = bench.replica_units(1000, world)
        buf = io.StringIO()

        class A:  # the reference arm's arguments
            workload, steps, warmup, cpu_blocks = "gauss_block", 1, 0, 1
        with redirect_stdout(buf):
            line = bench.run_reference(A)
        out.put((rank, slowest, units, line is not None))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_and_reference_arm():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    got = sorted(q.get() for _ in range(world))
    assert [g[1] for g in got] == [11.0, 11.0]        # max over ranks
    assert [g[2] for g in got] == [2000, 2000]        # every rank's replica counts
    assert [g[3] for g in got] == [True, False]       # only rank 0 runs the reference arm


def _spawned_rank():
    """What bench.py's self-started ranks see: the torchrun environment on a
    127.0.0.1 rendezvous, and a working process group across the ranks."""
    sys.path.insert(0, ROOT)
    import bench
    rank, local_rank, world = bench.dist_env()
    dist.init_process_group(bench.dist_backend(), rank=rank, world_size=world)
    try:
        return (rank, local_rank, world, bench.max_over_ranks(5.0 + rank), bench.replica_units(100, world),
                os.environ["MASTER_ADDR"])
    finally:
        dist.destroy_process_group()


def test_bench_starts_its_own_ranks_without_torchrun():
    """`bench.py --gpus N` outside torchrun starts N ranks itself (gloo on
    CPU here, NCCL on GPUs): each rank gets RANK = LOCAL_RANK, WORLD_SIZE = N,
    the job's time is the slowest rank's and its value counts every replica."""
    sys.path.insert(0, ROOT)
    import bench
    out = bench.spawn_ranks(2, _spawned_rank, (), backend="gloo", timeout=300)
    assert sorted(out) == [0, 1]
    for r, v in out.items():
        assert v == (r, r, 2, 6.0, 200, "127.0.0.1")


def test_single_process_defaults():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.replica_units(7, 1) == 7


def test_stored_traffic_follows_the_kernel_source():
    """A stored ncu traffic figure is reported only for the kernel source it
    was taken of: the AdamW call's hash covers both of its kernels' files."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.stored_traffic("no_such_workload", "sgd") is None
    hashes = {k: bench.kernel_source_hash(k) for k in bench.KERNEL_SOURCES}
    assert len(set(hashes.values())) == len(hashes)
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        stored = json.load(f)
    for workload, kernels in stored.items():
        for kernel, entry in kernels.items():
            got = bench.stored_traffic(workload, kernel)
            if entry["source_hash"] == hashes[kernel]:
                assert got == entry["bytes_per_launch"] > 0
            else:
                assert got is None
