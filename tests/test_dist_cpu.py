"""The benchmark's multi-rank host logic on CPU (gloo, world size 2).

Questions are independent, so under torchrun every rank scores its own
copy of the workload on its own GPU (replicas: no data exchange). The only
collective is the timing: the whole job runs as long as its slowest rank,
and the reported rate is all ranks' questions over that time. These tests
run two gloo ranks on the host to check exactly that, and that the
reference arm runs on rank 0 only.
"""
from __future__ import annotations

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        m = bench.reduce_max(times[rank])
        rate = bench.whole_job_rate(16384, m, world)
        ref_rc = None
        if rank != 0:
            class A:
                steps, warmup = 3, 3
            ref_rc = bench.run_reference(A())  # non-zero ranks leave without work
        q.put((rank, m, rate, ref_rc))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    times = [1.25, 2.5]  # ms per step on rank 0 and rank 1
    procs = [ctx.Process(target=_worker, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, m, rate, ref_rc in got:
        assert m == 2.5  # the slowest rank's time, on every rank
        assert rate == pytest.approx(2 * 16384 / 2.5e-3)
        if rank == 1:
            assert ref_rc == 0


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.0) == 3.0
    assert bench.whole_job_rate(100, 2.0, 1) == pytest.approx(50000.0)


def test_oracle_pool_counts_every_worker():
    """The CPU baseline's process pool (spawned workers, one sample each):
    every worker scores its own sample the asked number of times."""
    sys.path.insert(0, ROOT)
    import bench
    pool = bench.OraclePool(3, seed=1, workers=2)
    try:
        done, wall = pool.run(2)
    finally:
        pool.close()
    assert done == 2 * 3 * 2
    assert wall > 0.0
    assert bench._host_cores() >= 1


def test_kernel_fingerprint_ignores_comments_only():
    """The bench matches its ncu summary by a fingerprint of the kernel code:
    comments and blank lines do not change it, code does."""
    sys.path.insert(0, ROOT)
    import bench
    a = 'int x = 1; // note\n/* block\n comment */\n\nchar* s = "a // b";\n'
    b = 'int x = 1;\n\nchar* s = "a // b"; /* other note */\n'
    c = 'int x = 2;\nchar* s = "a // b";\n'
    assert bench._strip_comments(a) == bench._strip_comments(b) == 'int x = 1;\nchar* s = "a // b";'
    assert bench._strip_comments(c) != bench._strip_comments(a)
    assert len(bench._kernel_sha()) == 64
