"""Host side of the sharded data plane, on CPU: the z-slab partition, the
shards' slot ranges, and the exchange of every rank's layout and buffer
handle between two gloo ranks, checked against the oracle's plan (which
shards' halo slices each pulse writes into)."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from domain_decomposition_halo_build_gb300 import shard, synth  # noqa: E402


@pytest.mark.parametrize("grid,n", [((2, 4, 8), 1), ((2, 4, 8), 2), ((2, 4, 8), 3), ((2, 4, 8), 8),
                                    ((4, 4, 4), 4), ((5, 3, 7), 3), ((2, 2, 2), 2)])
def test_partition_is_contiguous_z_slabs(grid, n):
    parts = shard.partition(grid, n)
    nx, ny, nz = grid
    assert len(parts) == n
    assert parts[0][0] == 0 and sum(c for _, c in parts) == nx * ny * nz
    for (f0, c0), (f1, _) in zip(parts, parts[1:]):
        assert f0 + c0 == f1                       # contiguous id ranges
    for k, (first, count) in enumerate(parts):
        assert first % (nx * ny) == 0 and count % (nx * ny) == 0   # whole z layers
        assert count > 0
        for D in range(first, first + count):
            assert shard.shard_of_domain(grid, n, D) == k
            assert (k * nz) // n <= D // (nx * ny) < ((k + 1) * nz) // n


def test_partition_rejects_bad_counts():
    for n in (0, 3, 9):
        if n == 3:
            with pytest.raises(ValueError):
                shard.partition((4, 4, 2), n)     # more shards than z layers
            continue
        with pytest.raises(ValueError):
            shard.partition((2, 4, 8), n)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import oracle
    from domain_decomposition_halo_build_gb300 import shard as S, synth as Y
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = Y.WORKLOADS["water24k_2x4x8"]
        xyz, dom = Y.system(w)
        o = oracle.Oracle(w.box, w.grid, w.rc, xyz, dom)
        parts = S.partition(w.grid, world)
        ranges = S.slot_ranges(o.n_local, parts)
        first_domain, n_domains = parts[rank]
        first_slot, n_local = ranges[rank]
        layout = {"shard": rank, "first_domain": first_domain, "n_domains": n_domains,
                  "first_slot": first_slot, "n_local": n_local}
        handle = ("shard-buffer-of-rank-%d" % rank).encode()
        table = S.exchange_layouts(layout, handle)
        # the pulses this rank's domains send: where each destination slice lives
        cross = 0
        for s in range(first_domain, first_domain + n_domains):
            for p in range(o.n_pulses):
                info = o.pulse(s, p)
                if info.send_size == 0:
                    continue
                lo = int(o.base[info.recv_domain]) + info.atom_offset
                hi = lo + info.send_size - 1
                r0, r1 = S.owner_of_slot(table, lo), S.owner_of_slot(table, hi)
                assert r0 == r1 == S.shard_of_domain(w.grid, world, info.recv_domain)
                cross += r0 != rank
        out.put((rank, table, cross, o.n_local_total))
    finally:
        dist.destroy_process_group()


def test_layout_and_handle_exchange_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = sorted([q.get(timeout=300) for _ in ps], key=lambda t: t[0])
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    (_, t0, cross0, total), (_, t1, cross1, _) = res
    assert t0 == t1                                  # every rank holds the same table
    assert [t["shard"] for t in t0] == [0, 1]
    assert [t["handle"] for t in t0] == [b"shard-buffer-of-rank-0", b"shard-buffer-of-rank-1"]
    assert t0[0]["first_slot"] == 0 and t0[0]["n_local"] == t0[1]["first_slot"]
    assert t0[1]["first_slot"] + t0[1]["n_local"] == total       # the ranges tile the layout
    # z pulses cross the slab boundary (and the periodic wrap) in both directions
    assert cross0 > 0 and cross1 > 0
