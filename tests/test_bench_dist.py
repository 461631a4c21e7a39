"""Host-side logic of bench.py's N > 1 path, on CPU with gloo, world size 2.

Each rank is an independent replica; the only cross-rank steps are the
barrier and the maximum of the per-rank times.  The reference arm runs on
rank 0 alone."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r's times are (r+1) * base: the slowest rank must win
        local = [1.0 * (rank + 1), 0.25 * (rank + 1), 3.0 - rank]
        got = bench.max_over_ranks(local, "cpu", dist)
        dist.barrier()
        rate = bench.whole_job_rate(1000, world, got[0])
        out.put((rank, got, rate))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = [q.get(timeout=120) for _ in ps]
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, rate in res:
        assert got == [2.0, 0.5, 3.0]
        assert rate == pytest.approx(2 * 1000 / 2.0)


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2.5], "cpu", None) == [1.5, 2.5]


def test_reference_arm_non_zero_rank_exits_without_work(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")

    class A:
        workload = "water3k_2x1x1"
        steps = 1
        warmup = 0
        gpus = 2
    assert bench.run_reference(A()) == 0
    assert capsys.readouterr().out == ""


def test_replica_count_covers_the_l2():
    """The bench steps enough copies of a system that their data exceeds the
    L2 by the asked multiple: the 1M-atom system (about 100 MB with its
    tables) on a 135.5 MB L2 takes six copies; a system larger than the L2
    still takes two; a tiny one many."""
    sys.path.insert(0, ROOT)
    import bench
    l2 = 135_528_448
    per_1m = 24 * 1_831_410 + 68 * 831_410
    assert bench.replica_count(per_1m, l2) == 6
    assert bench.replica_count(per_1m, l2) * per_1m >= 4 * l2
    assert bench.replica_count(10 * l2, l2) == 2
    assert bench.replica_count(1_000_000, l2) == 543
