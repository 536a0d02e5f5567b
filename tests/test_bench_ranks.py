"""The multi-rank host logic of bench.py on CPU: two gloo ranks (replicas
only -- the attention path needs no exchange between GPUs, so the only
collective is the timing reduction).  Checks that every rank sees the
slowest rank's times, that the whole-job rate counts all ranks' bytes over
that time, and that the oracle arm leaves the work to rank 0."""
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


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        mine = [10.0 + rank, 5.0 - rank, 7.5]          # rank 1 is slower in the first value only
        got = bench._max_over_ranks(mine, "cpu")
        rate = bench._job_throughput(world, 1000.0, got[0])
        # the oracle arm: ranks other than 0 return at once, without output
        os.environ["RANK"], os.environ["WORLD_SIZE"] = str(rank), str(world)

        class A:  # the arguments run_reference reads
            workload, steps, warmup, sliding_window, attention_chunk, fp16 = 2, 3, 3, 0, 0, False
        skipped = bench.run_reference(A) is None if rank != 0 else True
        q.put((rank, got, rate, skipped))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, rate, skipped in res:
        assert got == [11.0, 5.0, 7.5]
        assert rate == pytest.approx(2 * 1000.0 / 11.0)
        assert skipped
