"""The bench's multi-process path, on CPU with the gloo backend (world size 2).

With --gpus N under torchrun every rank runs its own replica of the workload
(independent problems, no collective on the data path); the only collectives
are the barrier around the timed region and the max-over-ranks of the times.
These tests run exactly that host logic in two CPU processes.
"""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, local, w = bench.dist_env()
    assert (r, local, w) == (rank, rank, world)
    dist = bench.init_dist(w, "gloo")
    try:
        bench.barrier(dist)
        # each rank's mean step time; the job's time is the slowest rank's
        t = bench.max_over_ranks(1.0 + rank, dist)
        v = bench.aggregate_throughput(10.0, w, t)
        # the reference arm runs on rank 0 only; other ranks leave without work
        args = type("A", (), dict(workload=bench.HEADLINE, steps=1, warmup=0, gpus=w))()
        rc = bench.run_reference(args, rank, w) if rank != 0 else 0
        out[rank] = (t, v, rc)
        bench.barrier(dist)
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        t, v, rc = out[r]
        assert t == 2.0                     # max over ranks
        assert v == pytest.approx(10.0 * 2 / 2.0)  # all ranks' units over the slowest time
        assert rc == 0


def test_single_process_helpers():
    import bench
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.aggregate_throughput(8.0, 1, 2.0) == 4.0


def test_source_digest_ignores_comments_only():
    """A recorded ncu traffic figure stays valid across comment edits and is
    dropped (null) once the code of the kernel's sources changes."""
    import bench
    code = "int f(int x) {\n    return x + 1;  // add one\n}\n/* block\n   comment */\n"
    assert bench._code_only(code) == bench._code_only(code.replace("add one", "increment"))
    assert bench._code_only(code) == bench._code_only("// header\n" + code + "\n\n")
    assert bench._code_only(code) != bench._code_only(code.replace("x + 1", "x + 2"))
    assert "//" not in bench._code_only(code) and "/*" not in bench._code_only(code)


def test_recorded_traffic_lines_parse():
    """Every line of the committed traffic record names a known kernel and a
    positive byte count; a line whose digest no longer matches reads as None."""
    import os
    import bench
    path = os.path.join(bench.ROOT, "profiles", "ncu_traffic.txt")
    lines = [l.split() for l in open(path).read().splitlines() if l.strip() and not l.startswith("#")]
    assert lines
    for workload, kernel, digest, nbytes in lines:
        assert kernel in bench.KERNEL_SOURCES
        assert len(digest) == 16 and float(nbytes) > 0
        got = bench.recorded_traffic(workload, kernel)
        assert got is None or got == float(nbytes)
    assert bench.recorded_traffic("no_such_workload", "prefill_kernel") is None
