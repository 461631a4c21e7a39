"""The sharded data plane on one GPU: a plan's domains split into z-slabs,
each shard with its own buffer, the FUSED exchanges across the shards with
system-scope signals, every shard's work in one launch.  Compared bit for
bit with the oracle (the shards' buffers, put side by side, are the dense
local array)."""
import numpy as np
import pytest

import oracle
from domain_decomposition_halo_build_gb300 import shard, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _cat(shards):
    import torch
    return torch.cat(shards, 0).cpu().numpy()


def _case(name, n_shards, prune=False):
    import torch
    from domain_decomposition_halo_build_gb300 import halo
    w = synth.WORKLOADS[name]
    xyz, dom = synth.system(w)
    o = oracle.Oracle(w.box, w.grid, w.rc, xyz, dom, prune=prune)
    x = torch.from_numpy(xyz).cuda()
    d = torch.from_numpy(dom).cuda()
    plan = halo.HaloPlan(w.box, w.grid, w.rc, x, d, prune=prune)
    plan.shard(n_shards)
    return w, xyz, o, x, plan


@pytest.mark.parametrize("name,n", [("water24k_2x4x8", 1), ("water24k_2x4x8", 2),
                                    ("water24k_2x4x8", 3), ("water24k_2x4x8", 8),
                                    ("water48k_2x2x2", 2), ("water1M_4x4x4", 4)])
def test_sharded_exchanges_match_the_oracle(name, n):
    import torch
    w, xyz, o, x, plan = _case(name, n)
    try:
        parts = shard.partition(w.grid, n)
        ranges = shard.slot_ranges(o.n_local, parts)
        for k in range(n):
            lay = plan.shard_layout(k)
            assert (lay["first_domain"], lay["n_domains"]) == parts[k]
            assert (lay["first_slot"], lay["n_local"]) == ranges[k]
        want_x = o.load_home(xyz)
        o.exchange_x(want_x)
        f0 = synth.forces(o.n_local_total, seed=1)
        want_f = f0.copy()
        o.exchange_f(want_f)
        for call in range(2):
            xs = plan.load_home_sharded(x, plan.shard_buffers())
            plan.exchange_x_sharded(xs)
            fs = [torch.from_numpy(f0[a:a + c].copy()).cuda() for a, c in ranges]
            plan.exchange_f_sharded(fs)
            assert plan.status() == 0
            np.testing.assert_array_equal(_cat(xs).view(np.uint32), want_x.view(np.uint32),
                                          err_msg="coordinates, call %d" % call)
            np.testing.assert_array_equal(_cat(fs).view(np.uint32), want_f.view(np.uint32),
                                          err_msg="forces, call %d" % call)
        # store_home from the shards gives every atom's reduced force
        g = plan.store_home_sharded(fs)
        l2g = o.local_to_global()
        home = np.concatenate([np.arange(o.base[D], o.base[D] + o.n_home[D]) for D in range(o.n_domains)])
        want_g = np.zeros((o.n_atoms, 3), np.float32)
        want_g[l2g[home]] = want_f[home]
        np.testing.assert_array_equal(g.cpu().numpy(), want_g)
    finally:
        plan.close()


def test_sharded_and_dense_calls_interleave():
    """Dense FUSED and sharded calls on one plan share its counters and
    tickets; each result still equals the oracle's."""
    import torch
    w, xyz, o, x, plan = _case("water24k_2x4x8", 4)
    try:
        plan.set_mode("fused")
        want = o.load_home(xyz)
        o.exchange_x(want)
        for call in range(3):
            loc = plan.load_home(x)
            plan.exchange_x(loc)
            xs = plan.load_home_sharded(x, plan.shard_buffers())
            plan.exchange_x_sharded(xs)
            assert plan.status() == 0
            assert np.array_equal(loc.cpu().numpy(), want)
            assert np.array_equal(_cat(xs), want)
    finally:
        plan.close()


@pytest.mark.parametrize("n", [1, 2])
def test_sharding_survives_rebuild_and_pruning(n):
    import torch
    w = synth.WORKLOADS["water24k_2x4x8"]
    xyz, dom = synth.system(w)
    from domain_decomposition_halo_build_gb300 import halo
    x = torch.from_numpy(xyz).cuda()
    d = torch.from_numpy(dom).cuda()
    plan = halo.HaloPlan(w.box, w.grid, w.rc, x, d, prune=True)
    try:
        plan.set_mode("flat")          # the sharded calls run on their own work lists
        plan.shard(n)
        x2, d2 = synth.displaced(xyz, w.box, w.grid, 1)
        plan.rebuild(torch.from_numpy(x2).cuda(), torch.from_numpy(d2).cuda())
        o = oracle.Oracle(w.box, w.grid, w.rc, x2, d2, prune=True)
        want = o.load_home(x2)
        o.exchange_x(want)
        xs = plan.load_home_sharded(torch.from_numpy(x2).cuda(), plan.shard_buffers())
        plan.exchange_x_sharded(xs)
        assert plan.status() == 0
        assert np.array_equal(_cat(xs), want)
    finally:
        plan.close()


def test_shard_counts_and_pointers_are_checked():
    import ctypes
    import torch
    from domain_decomposition_halo_build_gb300 import halo
    w = synth.WORKLOADS["water3k_2x1x1"]            # one z layer: one shard only
    xyz, dom = synth.system(w)
    plan = halo.HaloPlan(w.box, w.grid, w.rc, torch.from_numpy(xyz).cuda(),
                         torch.from_numpy(dom).cuda())
    try:
        lib = halo.load_library()
        for n in (0, 2, 9):
            assert lib.halo_shard(plan.handle, n, None) == halo.EINVAL
        plan.shard(1)
        ptrs = (ctypes.c_void_p * 1)(None)
        assert lib.halo_exchange_x_sharded(plan.handle, ptrs, None) == halo.EINVAL
        assert lib.halo_shard_layout(plan.handle, 1, None, None, None, None) == halo.EINVAL
    finally:
        plan.close()


def test_sharded_wait_times_out_and_recovers():
    """A dropped producer signal in the sharded coordinate exchange: the
    system-scope waits give up after 50 ms, HALO_ETIMEOUT, then exact."""
    from domain_decomposition_halo_build_gb300 import halo
    w, xyz, o, x, plan = _case("water24k_2x4x8", 2)
    try:
        plan.set_wait_timeout(0.05)
        plan.debug_drop_signal(0, 0)
        xs = plan.load_home_sharded(x, plan.shard_buffers())
        plan.exchange_x_sharded(xs)
        assert plan.status() == halo.ETIMEOUT
        want = o.load_home(xyz)
        o.exchange_x(want)
        xs = plan.load_home_sharded(x, plan.shard_buffers())
        plan.exchange_x_sharded(xs)
        assert plan.status() == halo.OK
        assert np.array_equal(_cat(xs), want)
    finally:
        plan.close()
