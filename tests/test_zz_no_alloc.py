"""halo_exchange_x_noalloc: the coordinate exchange for callers that may not
allocate device memory when they call in (a host framework whose pool
allocator owns all device memory, or a latency-critical loop where cudaMalloc
/ cudaFree and the device-wide synchronisation they can cause are not
acceptable).  Its scratch is a fixed array inside the library, whose device
address halo_setup looks up.

Checked through the C ABI:
- two calls in a row give the oracle's coordinates and halo_exchange_x's,
  bit-exact (the tolerance of every coordinate test here);
- calls interleaved with halo_exchange_x on one plan (two epoch schemes: the
  plan's growing ticket, and the fixed array cleared on every call) leave
  each other's results intact;
- a call whose wait times out (a dropped signal, 50 ms limit) is reported by
  halo_status, and the next call is exact again;
- a plan too large for the fixed array is refused with HALO_ESCRATCH;
- the calls, the first one included, leave the device's free memory
  unchanged (a coarse guard: free memory is counted in whole driver pages).
This file is collected last and builds everything it needs, so it runs alone
or after the other tests."""
import ctypes

import numpy as np
import pytest

import oracle
from domain_decomposition_halo_build_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _plan(name):
    import torch
    from domain_decomposition_halo_build_gb300 import halo
    w = synth.WORKLOADS[name]
    xyz, dom = synth.system(w)
    x = torch.from_numpy(xyz).cuda()
    d = torch.from_numpy(dom).cuda()
    return halo.HaloPlan(w.box, w.grid, w.rc, x, d), x


@pytest.mark.parametrize("name", ["water24k_2x4x8", "water1M_4x4x4"])
def test_noalloc_matches_exchange_x_twice(name):
    import torch
    from domain_decomposition_halo_build_gb300 import halo
    lib = halo.load_library()
    plan, x = _plan(name)
    try:
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        want = plan.load_home(x)
        assert lib.halo_exchange_x(plan.handle, ctypes.c_void_p(want.data_ptr()), stream) == 0
        assert plan.status() == 0
        want = want.cpu().numpy()
        for call in range(2):
            got = plan.load_home(x)
            got_ptr = ctypes.c_void_p(got.data_ptr())
            assert lib.halo_exchange_x_noalloc(plan.handle, got_ptr, stream) == halo.OK
            assert plan.status() == halo.OK
            np.testing.assert_array_equal(got.cpu().numpy().view(np.uint32), want.view(np.uint32),
                                          err_msg="call %d" % call)
    finally:
        plan.close()


def _oracle_x(name):
    w = synth.WORKLOADS[name]
    xyz, dom = synth.system(w)
    o = oracle.Oracle(w.box, w.grid, w.rc, xyz, dom)
    want = o.load_home(xyz)
    o.exchange_x(want)
    return want


def test_noalloc_matches_the_oracle_twice():
    """Directly against the CPU oracle, on the multi-pulse system whose
    forwarded entries wait on earlier pulses: two calls in a row."""
    import torch
    from domain_decomposition_halo_build_gb300 import halo
    lib = halo.load_library()
    want = _oracle_x("water24k_2x4x8")
    plan, x = _plan("water24k_2x4x8")
    try:
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        for call in range(2):
            got = plan.load_home(x)
            assert lib.halo_exchange_x_noalloc(plan.handle, ctypes.c_void_p(got.data_ptr()),
                                               stream) == halo.OK
            assert plan.status() == halo.OK
            np.testing.assert_array_equal(got.cpu().numpy().view(np.uint32), want.view(np.uint32),
                                          err_msg="call %d" % call)
    finally:
        plan.close()


def test_noalloc_interleaved_with_exchange_x():
    """x, noalloc, x, noalloc on one plan, each result against the oracle."""
    import torch
    from domain_decomposition_halo_build_gb300 import halo
    lib = halo.load_library()
    want = _oracle_x("water24k_2x4x8")
    plan, x = _plan("water24k_2x4x8")
    try:
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        for call, fn in enumerate([lib.halo_exchange_x, lib.halo_exchange_x_noalloc] * 2):
            got = plan.load_home(x)
            assert fn(plan.handle, ctypes.c_void_p(got.data_ptr()), stream) == halo.OK
            assert plan.status() == halo.OK
            np.testing.assert_array_equal(got.cpu().numpy().view(np.uint32), want.view(np.uint32),
                                          err_msg="call %d" % call)
    finally:
        plan.close()


def test_noalloc_after_a_timed_out_wait():
    """A producer's signal dropped on the host side (test hook) makes the
    call's consumers give up after 50 ms; halo_status reports HALO_ETIMEOUT
    and clears it, and the next call is exact again.  No GPU fault: every
    wait is bounded."""
    import torch
    from domain_decomposition_halo_build_gb300 import halo
    lib = halo.load_library()
    want = _oracle_x("water24k_2x4x8")
    plan, x = _plan("water24k_2x4x8")
    try:
        plan.set_wait_timeout(0.05)
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        plan.debug_drop_signal(0, 0)   # z0 of domain 0 feeds the z1 pulse of its receiver
        loc = plan.load_home(x)
        assert lib.halo_exchange_x_noalloc(plan.handle, ctypes.c_void_p(loc.data_ptr()),
                                           stream) == halo.OK
        assert plan.status() == halo.ETIMEOUT
        assert plan.status() == halo.OK
        for call in range(2):
            got = plan.load_home(x)
            assert lib.halo_exchange_x_noalloc(plan.handle, ctypes.c_void_p(got.data_ptr()),
                                               stream) == halo.OK
            assert plan.status() == halo.OK
            np.testing.assert_array_equal(got.cpu().numpy().view(np.uint32), want.view(np.uint32),
                                          err_msg="call %d after the timeout" % call)
    finally:
        plan.close()


def test_noalloc_leaves_free_memory_unchanged():
    """From before the first call on the plan: halo_setup placed the fixed
    array, so no call here allocates."""
    import torch
    from domain_decomposition_halo_build_gb300 import halo
    lib = halo.load_library()
    plan, x = _plan("water24k_2x4x8")
    try:
        loc = plan.load_home(x)
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        ptr = ctypes.c_void_p(loc.data_ptr())
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        for _ in range(6):
            assert lib.halo_exchange_x_noalloc(plan.handle, ptr, stream) == 0
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0
        assert plan.status() == 0
    finally:
        plan.close()


def test_noalloc_refuses_plans_beyond_the_fixed_array():
    import torch
    from domain_decomposition_halo_build_gb300 import halo
    lib = halo.load_library()
    box, grid, rc = (8.0, 8.0, 8.0), (16, 16, 16), 1.4      # 4096 domains x 9 pulses
    xyz, dom = synth.custom_system(40000, box, grid, seed=8)
    x = torch.from_numpy(xyz).cuda()
    d = torch.from_numpy(dom).cuda()
    plan = halo.HaloPlan(box, grid, rc, x, d)
    try:
        assert plan.n_domains * plan.n_pulses > halo.NOALLOC_MAX_COUNTERS
        loc = plan.load_home(x)
        before = loc.clone()
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        code = lib.halo_exchange_x_noalloc(plan.handle, ctypes.c_void_p(loc.data_ptr()), stream)
        assert code == halo.ESCRATCH
        assert "fixed scratch" in halo.strerror(code)
        torch.cuda.synchronize()
        assert torch.equal(loc, before)                       # nothing ran
    finally:
        plan.close()


def test_noalloc_needs_the_fused_work_lists():
    """A plan rebuilt in FLAT mode has no FUSED work lists (a rebuild builds
    only the current mode's tables), and building them would allocate: the
    call refuses with HALO_EINVAL and touches nothing.  After
    halo_set_mode(FUSED) it runs and matches halo_exchange_x."""
    import torch
    from domain_decomposition_halo_build_gb300 import halo
    lib = halo.load_library()
    plan, x = _plan("water24k_2x4x8")
    try:
        d = torch.from_numpy(synth.system(synth.WORKLOADS["water24k_2x4x8"])[1]).cuda()
        plan.set_mode("flat")
        plan.rebuild(x, d)
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        loc = plan.load_home(x)
        before = loc.clone()
        code = lib.halo_exchange_x_noalloc(plan.handle, ctypes.c_void_p(loc.data_ptr()), stream)
        assert code == halo.EINVAL
        torch.cuda.synchronize()
        assert torch.equal(loc, before)
        plan.set_mode("fused")
        want = plan.load_home(x)
        plan.exchange_x(want)
        assert lib.halo_exchange_x_noalloc(plan.handle, ctypes.c_void_p(loc.data_ptr()), stream) == 0
        assert plan.status() == 0
        assert torch.equal(loc.view(torch.int32), want.view(torch.int32))
    finally:
        plan.close()
