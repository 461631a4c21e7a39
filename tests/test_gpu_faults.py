"""Failure detection without a GPU fault: a producer's completion signal is
suppressed on the host side (test hook), its consumers' bounded waits run out
after a short limit, the kernel returns, and the plan reports HALO_ETIMEOUT
through halo_status(); the context stays usable and the next exchange is
correct."""
import numpy as np
import pytest

import oracle
from domain_decomposition_halo_build_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def test_dropped_signal_times_out_and_recovers():
    import torch
    from domain_decomposition_halo_build_gb300 import halo
    w = synth.WORKLOADS["water24k_2x4x8"]
    xyz, dom = synth.system(w)
    o = oracle.Oracle(w.box, w.grid, w.rc, xyz, dom)
    x = torch.from_numpy(xyz).cuda()
    d = torch.from_numpy(dom).cuda()
    plan = halo.HaloPlan(w.box, w.grid, w.rc, x, d)
    try:
        plan.set_wait_timeout(0.05)
        # pulse 0 (z0) of domain 0 feeds the whole z1 pulse of its receiver
        plan.debug_drop_signal(0, 0)
        loc = plan.load_home(x)
        plan.exchange_x(loc)
        assert plan.status() == halo.ETIMEOUT
        assert plan.status() == halo.OK          # cleared
        want = o.load_home(xyz)
        o.exchange_x(want)
        for _ in range(3):                       # flags were reset: exchanges work again
            loc = plan.load_home(x)
            plan.exchange_x(loc)
            assert plan.status() == halo.OK
            np.testing.assert_array_equal(loc.cpu().numpy(), want)
    finally:
        plan.close()


def test_bad_arguments_return_codes():
    import ctypes
    from domain_decomposition_halo_build_gb300 import halo
    lib = halo.load_library()
    assert lib.halo_exchange_x(None, None, None) == halo.EINVAL
    assert lib.halo_status(None, None) == halo.EINVAL
    assert lib.halo_set_wait_timeout(None, 1.0) == halo.EINVAL
    h = ctypes.c_void_p()
    box = (ctypes.c_float * 3)(1, 1, 1)
    grid = (ctypes.c_int32 * 3)(1, 1, 1)
    assert lib.halo_setup(box, grid, ctypes.c_float(0.1), None, None, 10, None,
                          ctypes.byref(h)) == halo.EINVAL


def test_failed_rebuild_refuses_exchanges_until_rebuilt():
    import torch
    from domain_decomposition_halo_build_gb300 import halo
    w = synth.WORKLOADS["water48k_2x2x2"]
    xyz, dom = synth.system(w)
    x = torch.from_numpy(xyz).cuda()
    d = torch.from_numpy(dom).cuda()
    plan = halo.HaloPlan(w.box, w.grid, w.rc, x, d)
    try:
        loc = plan.load_home(x)
        bad = d.clone()
        bad[123] = 99                                   # domain id out of range
        with pytest.raises(halo.HaloError) as e:
            plan.rebuild(x, bad)
        assert e.value.code == halo.EDOMAIN
        with pytest.raises(halo.HaloError) as e:
            plan.exchange_x(loc)
        assert e.value.code == halo.EINVAL
        with pytest.raises(halo.HaloError) as e:        # so do the plan queries
            plan.pulse(0, 0)
        assert e.value.code == halo.EINVAL
        plan.rebuild(x, d)                              # a good rebuild restores it
        loc = plan.load_home(x)
        plan.exchange_x(loc)
        assert plan.status() == halo.OK
        o = oracle.Oracle(w.box, w.grid, w.rc, xyz, dom)
        want = o.load_home(xyz)
        o.exchange_x(want)
        np.testing.assert_array_equal(loc.cpu().numpy(), want)
    finally:
        plan.close()


def test_build_buffer_overflow_is_detected_and_retried():
    """A build buffer far too small for the halo (test hook): the pulse kernels
    stop writing at its end, the build detects the overflow, grows the buffer
    and runs again; the result is the oracle's."""
    import torch
    from domain_decomposition_halo_build_gb300 import halo
    w = synth.WORKLOADS["water24k_2x4x8"]
    xyz, dom = synth.system(w)
    x = torch.from_numpy(xyz).cuda()
    d = torch.from_numpy(dom).cuda()
    plan = halo.HaloPlan(w.box, w.grid, w.rc, x, d)
    try:
        assert plan.build_attempts == 1
        plan.debug_set_build_capacity(w.n_atoms + 100)     # room for 100 halo slots
        plan.rebuild(x, d)
        assert plan.build_attempts > 1
        o = oracle.Oracle(w.box, w.grid, w.rc, xyz, dom)
        assert plan.n_local_total == o.n_local_total
        maps, offs = plan.index_maps()
        for p in range(o.n_pulses):
            for s in range(o.n_domains):
                want = o.index_map(s, p)
                got = maps[offs[p * o.n_domains + s]:offs[p * o.n_domains + s + 1]]
                np.testing.assert_array_equal(got, want)
        loc = plan.load_home(x)
        plan.exchange_x(loc)
        assert plan.status() == halo.OK
        want = o.load_home(xyz)
        o.exchange_x(want)
        np.testing.assert_array_equal(loc.cpu().numpy(), want)
        with pytest.raises(halo.HaloError):
            plan.debug_set_build_capacity(0)
    finally:
        plan.close()


def test_wait_timeout_from_the_environment(monkeypatch):
    """HALO_WAIT_TIMEOUT_MS sets a new plan's wait limit: with 30 ms a dropped
    signal ends the exchange well before the 1 s default could."""
    import time
    import torch
    from domain_decomposition_halo_build_gb300 import halo
    monkeypatch.setenv("HALO_WAIT_TIMEOUT_MS", "30")
    w = synth.WORKLOADS["water24k_2x4x8"]
    xyz, dom = synth.system(w)
    x = torch.from_numpy(xyz).cuda()
    d = torch.from_numpy(dom).cuda()
    plan = halo.HaloPlan(w.box, w.grid, w.rc, x, d)
    try:
        loc = plan.load_home(x)
        torch.cuda.synchronize()
        plan.debug_drop_signal(0, 0)
        t0 = time.perf_counter()
        plan.exchange_x(loc)
        code = plan.status()
        elapsed = time.perf_counter() - t0
        assert code == halo.ETIMEOUT
        assert elapsed < 0.6, elapsed
        plan.exchange_x(loc)
        assert plan.status() == halo.OK
    finally:
        plan.close()
