"""The multi-replica path of bench.py on CPU (gloo, world size 2).

Every run here has one GPU, so N > 1 means N independent replicas: each rank
times its own steps, the job's step time is the slowest rank's (maximum over
ranks), and the reported throughput counts every rank's bytes.  These tests
run that reduction over a real two-process gloo group, and check that
non-zero ranks of the reference arm leave without doing work.
"""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        r, w, local = bench.dist_env()
        # rank 0 is faster on the first timing, rank 1 on the second
        vals = bench.reduce_max_over_ranks([1.0 + rank, 10.0 - rank, 0.5], w, "cpu")
        q.put((rank, r, w, local, vals, bench.aggregate_gbs(4e9, w, vals[0])))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0, 0]
    for rank, r, w, local, vals, gbs in got:
        assert (r, w, local) == (rank, 2, rank)
        assert vals == [2.0, 10.0, 0.5]  # the maximum of each timing over both ranks
        assert gbs == pytest.approx(2 * 4e9 / 2e-3 / 1e9)  # both replicas' bytes in 2 ms


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.reduce_max_over_ranks([3, 1.5], 1, "cpu") == [3.0, 1.5]
    assert bench.aggregate_gbs(1e9, 1, 1.0) == pytest.approx(1000.0)


def test_reference_arm_nonzero_rank_exits_without_work(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2"])
    out = io.StringIO()
    with redirect_stdout(out):
        bench.main()
    assert out.getvalue() == ""
