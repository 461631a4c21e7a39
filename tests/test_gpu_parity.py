"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bar: index maps, splits, sizes, offsets, shifts, local-to-global ids and
exchanged coordinates bit-exact; forces bit-exact (the kernel keeps the
oracle's per-slot add order), and in any case within 1e-6 relative per fp32
component.
"""
import numpy as np
import pytest

import oracle
import pins
from domain_decomposition_halo_build_gb300 import synth

pytestmark = pytest.mark.gpu

FORCE_RTOL = 1e-6


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def gpu_plan(box, grid, rc, xyz, dom, prune=False):
    from gpu_adaptor import GpuPlan
    return GpuPlan(box, grid, rc, xyz, dom, prune=prune)


def bits(a):
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


def compare_plans(g, o):
    assert g.n_pulses == o.n_pulses
    np.testing.assert_array_equal(g.pulse_dim, o.pulse_dim)
    np.testing.assert_array_equal(g.pulses_per_dim, o.pulses_per_dim)
    np.testing.assert_array_equal(g.n_home, o.n_home)
    np.testing.assert_array_equal(g.n_local, o.n_local)
    np.testing.assert_array_equal(g.base, o.base)
    assert g.n_local_total == o.n_local_total
    maps, offs = g.plan.index_maps()
    nd = o.n_domains
    for p in range(o.n_pulses):
        for s in range(nd):
            gi, oi = g.pulse(s, p), o.pulse(s, p)
            for k in ("recv_domain", "send_size", "split", "dep_offset", "atom_offset"):
                assert getattr(gi, k) == getattr(oi, k), ((s, p), k)
            np.testing.assert_array_equal(bits(gi.coord_shift), bits(oi.coord_shift))
            want = o.index_map(s, p)
            got = maps[offs[p * nd + s]:offs[p * nd + s + 1]]
            np.testing.assert_array_equal(got, want, err_msg=str((s, p)))
    np.testing.assert_array_equal(g.local_to_global(), o.local_to_global())


def compare_exchanges(g, o, xyz, reps=2, seed=1):
    want_x = o.load_home(xyz)
    o.exchange_x(want_x)
    for _ in range(reps):
        got = g.load_home(xyz)
        g.exchange_x(got)
        np.testing.assert_array_equal(bits(got), bits(want_x), err_msg="coordinates")
    f0 = synth.forces(o.n_local_total, seed=seed)
    want = f0.copy()
    got = f0.copy()
    for r in range(reps):
        o.exchange_f(want)
        g.exchange_f(got)
        rel = np.abs(got.astype(np.float64) - want) / np.maximum(np.abs(want.astype(np.float64)), 1e-30)
        assert float(rel.max()) <= FORCE_RTOL, ("force rel err", float(rel.max()), r)
        np.testing.assert_array_equal(bits(got), bits(want), err_msg="forces (bit-exact)")


WORKLOADS = list(synth.WORKLOADS)


@pytest.fixture(scope="module")
def cases():
    cache = {}

    def get(name):
        if name not in cache:
            w = synth.WORKLOADS[name]
            xyz, dom = synth.system(w)
            o = oracle.Oracle(w.box, w.grid, w.rc, xyz, dom)
            cache[name] = (w, xyz, dom, o, gpu_plan(w.box, w.grid, w.rc, xyz, dom))
        return cache[name]

    yield get
    for v in cache.values():
        v[4].close()


@pytest.mark.parametrize("name", pins.EXAMPLES)
def test_golden_examples_on_gpu(name):
    """The hand-worked examples, run through the library."""
    pins.check_example(gpu_plan, pins.load_example(name))


@pytest.mark.parametrize("name", WORKLOADS)
def test_plan_parity(cases, name):
    w, xyz, dom, o, g = cases(name)
    compare_plans(g, o)


MODES = ["fused", "stepwise", "flat", "staged"]
# staged synchronises the host inside every call, which stream capture forbids
GRAPH_MODES = ["fused", "stepwise", "flat"]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("name", WORKLOADS)
def test_exchange_parity(cases, name, mode):
    w, xyz, dom, o, g = cases(name)
    g.plan.set_mode(mode)
    try:
        assert g.plan.mode == mode
        compare_exchanges(g, o, xyz)
    finally:
        g.plan.set_mode("fused")


@pytest.mark.parametrize("name", ["water24k_2x4x8", "water1M_4x4x4"])
def test_gpu_forces_integer_closed_form(cases, name):
    w, xyz, dom, o, g = cases(name)
    pins.check_forces_integer(g)


def test_rebuild_after_displacement(cases):
    """3M-atom system: displace by N(0, 0.01 nm), rebuild (twice, the second time
    with the flat mode active, whose tables are rebuilt too), compare again."""
    w, xyz, dom, o, g = cases("water3M_8x8x8")
    for k, mode in ((1, "fused"), (2, "flat")):
        g.plan.set_mode(mode)
        xk, dk = synth.displaced(xyz, w.box, w.grid, k=k)
        g.rebuild(xk, dk)
        assert g.plan.mode == mode
        ok = oracle.Oracle(w.box, w.grid, w.rc, xk, dk)
        compare_plans(g, ok)
        compare_exchanges(g, ok, xk, reps=1)
    # the cached plan serves other tests: back to the original positions
    g.plan.set_mode("fused")
    g.rebuild(xyz, dom)
    compare_plans(g, o)


def test_mode_tables_after_a_rebuild_in_each_mode():
    """A setup or rebuild builds only the current mode's tables; selecting
    another mode afterwards builds its own (FUSED work lists, FLAT tables,
    STAGED buffer).  After a rebuild in each mode of the multi-pulse system,
    every mode matches the oracle of the displaced positions."""
    w = synth.WORKLOADS["water24k_2x4x8"]
    xyz, dom = synth.system(w)
    g = gpu_plan(w.box, w.grid, w.rc, xyz, dom)
    try:
        for k, mode_a in enumerate(MODES, start=1):
            g.plan.set_mode(mode_a)
            xk, dk = synth.displaced(xyz, w.box, w.grid, k=k)
            g.rebuild(xk, dk)
            assert g.plan.mode == mode_a
            ok = oracle.Oracle(w.box, w.grid, w.rc, xk, dk)
            compare_plans(g, ok)
            for mode_b in MODES:
                g.plan.set_mode(mode_b)
                compare_exchanges(g, ok, xk, reps=1)
    finally:
        g.plan.close()


@pytest.mark.parametrize("mode", ["fused", "flat"])
def test_bound_exchange_matches_the_checked_calls(mode):
    """HaloPlan.bind: the same C calls with the tensor checks done once.  Bit
    for bit the same results; wrong shapes refused at bind time; calls after
    a rebuild that changed the slot count, or after close, refused."""
    import torch
    from domain_decomposition_halo_build_gb300 import halo
    w = synth.WORKLOADS["water24k_2x4x8"]
    xyz, dom = synth.system(w)
    x = torch.from_numpy(xyz).cuda()
    d = torch.from_numpy(dom).cuda()
    plan = halo.HaloPlan(w.box, w.grid, w.rc, x, d)
    try:
        plan.set_mode(mode)
        f0 = torch.from_numpy(synth.forces(plan.n_local_total, seed=6)).cuda()
        want_x = plan.load_home(x)
        plan.exchange_x(want_x)
        want_f = f0.clone()
        plan.exchange_f(want_f)
        loc, f = plan.load_home(x), f0.clone()
        b = plan.bind(loc, f)
        b.x()
        b.f()
        assert plan.status() == 0
        assert torch.equal(loc.view(torch.int32), want_x.view(torch.int32))
        assert torch.equal(f.view(torch.int32), want_f.view(torch.int32))
        with pytest.raises(ValueError):
            plan.bind(loc[:-1])
        with pytest.raises(ValueError):
            plan.bind(None, f).x()
        xk, dk = synth.displaced(xyz, w.box, w.grid, k=3)
        plan.rebuild(torch.from_numpy(xk).cuda(), torch.from_numpy(dk).cuda())
        if plan.n_local_total != loc.shape[0]:
            with pytest.raises(halo.HaloError):
                b.x()
    finally:
        plan.close()
    with pytest.raises(halo.HaloError):
        b.f()


EDGE = [
    # (box, grid, rc, n_atoms, seed)
    ((2.0, 2.0, 2.0), (1, 1, 1), 0.5, 37, 0),        # one domain, no pulses
    ((3.0, 3.0, 3.0), (2, 1, 1), 0.5, 1, 0),         # a single atom
    ((2.4, 2.4, 2.4), (3, 3, 3), 1.0, 3000, 3),      # two pulses in every dim
    ((3.2, 3.2, 3.2), (4, 1, 1), 1.0, 777, 4),       # 1D, two pulses, ragged
    ((4.0, 4.0, 4.0), (1, 2, 5), 1.1, 1500, 5),      # x undecomposed
    ((5.0, 4.0, 3.0), (5, 4, 3), 0.9, 20000, 6),     # rectangular box, odd grid
    ((6.0, 6.0, 6.0), (3, 3, 3), 0.05, 2000, 7),     # almost nothing sent
    ((8.0, 8.0, 8.0), (16, 16, 16), 1.4, 40000, 8),  # 4096 domains, 3 pulses per dim
    ((10.0, 8.0, 8.0), (10, 8, 8), 0.9, 30000, 9),   # 640 domains: 2048-atom partition tiles
]


@pytest.mark.parametrize("box,grid,rc,n,seed", EDGE)
def test_edge_cases(box, grid, rc, n, seed):
    xyz, dom = synth.custom_system(n, box, grid, seed=seed)
    o = oracle.Oracle(box, grid, rc, xyz, dom)
    g = gpu_plan(box, grid, rc, xyz, dom)
    try:
        compare_plans(g, o)
        for mode in MODES:
            g.plan.set_mode(mode)
            compare_exchanges(g, o, xyz)
    finally:
        g.close()


def test_empty_domains_and_skewed_load():
    """All atoms in two of 27 domains: most senders send nothing."""
    box, grid, rc = (3.0, 3.0, 3.0), (3, 3, 3), 0.7
    rng = np.random.default_rng(9)
    xyz = (rng.random((5000, 3)) * np.array([0.9, 0.9, 2.9])).astype(np.float32)
    dom = synth.assign_domains(xyz, box, grid)
    o = oracle.Oracle(box, grid, rc, xyz, dom)
    g = gpu_plan(box, grid, rc, xyz, dom)
    try:
        assert (o.n_home == 0).sum() >= 20
        compare_plans(g, o)
        for mode in MODES:
            g.plan.set_mode(mode)
            compare_exchanges(g, o, xyz)
    finally:
        g.close()


@pytest.mark.parametrize("name", ["water24k_2x4x8", "water48k_2x2x2"])
def test_unaligned_inputs(name):
    """Coordinates and domain ids that start 12 and 4 bytes past a 16-byte
    boundary (views one atom into larger arrays): the home partition copies
    its tiles with plain loads instead of 16-byte copies."""
    import torch
    w = synth.WORKLOADS[name]
    xyz, dom = synth.system(w)
    o = oracle.Oracle(w.box, w.grid, w.rc, xyz, dom)
    g = gpu_plan(w.box, w.grid, w.rc, xyz, dom)
    try:
        xs = torch.zeros((len(xyz) + 1, 3), dtype=torch.float32, device="cuda")
        ds = torch.zeros(len(dom) + 1, dtype=torch.int32, device="cuda")
        xs[1:] = torch.from_numpy(xyz)
        ds[1:] = torch.from_numpy(dom)
        x, d = xs[1:], ds[1:]
        assert x.data_ptr() % 16 != 0 and d.data_ptr() % 16 != 0
        g.plan.rebuild(x, d)
        g._sync()
        compare_plans(g, o)
        g.plan.set_mode("flat")
        compare_exchanges(g, o, xyz)
    finally:
        g.close()


def test_copied_readbacks(monkeypatch):
    """With HALO_STAGE_COPIES set at setup the build's readbacks are copied
    instead of written into mapped host memory by the last kernels: the same
    plan, tables and exchanges, through a rebuild, in FUSED and FLAT mode."""
    monkeypatch.setenv("HALO_STAGE_COPIES", "1")
    w = synth.WORKLOADS["water24k_2x4x8"]
    xyz, dom = synth.system(w)
    g = gpu_plan(w.box, w.grid, w.rc, xyz, dom)
    try:
        o = oracle.Oracle(w.box, w.grid, w.rc, xyz, dom)
        compare_plans(g, o)
        compare_exchanges(g, o, xyz)                  # FUSED (the default)
        g.plan.set_mode("flat")
        compare_exchanges(g, o, xyz)
        x2, d2 = synth.displaced(xyz, w.box, w.grid, 3)
        g.rebuild(x2, d2)
        o2 = oracle.Oracle(w.box, w.grid, w.rc, x2, d2)
        compare_plans(g, o2)
        compare_exchanges(g, o2, x2)
    finally:
        g.close()


def test_setup_errors():
    import torch
    from domain_decomposition_halo_build_gb300 import halo
    xyz, dom = synth.custom_system(100, (3, 3, 3), (3, 1, 1), seed=1)
    x = torch.from_numpy(xyz).cuda()
    d = torch.from_numpy(dom).cuda()
    with pytest.raises(halo.HaloError) as e:
        halo.HaloPlan((3, 3, 3), (3, 1, 1), 2.5, x, d)
    assert e.value.code == halo.EPULSES
    bad = d.clone()
    bad[7] = 3
    with pytest.raises(halo.HaloError) as e:
        halo.HaloPlan((3, 3, 3), (3, 1, 1), 0.5, x, bad)
    assert e.value.code == halo.EDOMAIN
    with pytest.raises(halo.HaloError) as e:
        halo.HaloPlan((3, 3, 3), (3, 1, 1), 0.0, x, d)
    assert e.value.code == halo.EINVAL
    with pytest.raises(halo.HaloError) as e:
        halo.HaloPlan((3, 3, 3), (0, 1, 1), 0.5, x, d)
    assert e.value.code == halo.EINVAL


@pytest.mark.parametrize("mode", MODES)
def test_launches_per_direction(cases, mode):
    """fused and flat: one launch per direction; stepwise: one per pulse;
    staged: two per pulse (pack and transfer, or transfer and unpack)."""
    w, xyz, dom, o, g = cases("water24k_2x4x8")
    g.plan.set_mode(mode)
    try:
        x0, f0 = g.plan.launch_counts()
        loc = g.plan.load_home(g.xyz_d)
        g.plan.exchange_x(loc)
        g.plan.exchange_f(loc)
        assert g.plan.status() == 0
        x1, f1 = g.plan.launch_counts()
        want = {"stepwise": g.n_pulses, "staged": 2 * g.n_pulses}.get(mode, 1)
        assert (x1 - x0, f1 - f0) == (want, want)
    finally:
        g.plan.set_mode("fused")


def test_determinism_repeated(cases):
    """Twenty back-to-back x+f exchanges give bitwise identical results (a race
    would show up as run-to-run variance)."""
    import torch
    w, xyz, dom, o, g = cases("water48k_2x2x2")
    f0 = torch.from_numpy(synth.forces(g.n_local_total, seed=3)).cuda()
    ref = None
    for _ in range(20):
        loc = g.plan.load_home(g.xyz_d)
        g.plan.exchange_x(loc)
        f = f0.clone()
        g.plan.exchange_f(f)
        out = (loc.cpu().numpy().view(np.uint32).copy(), f.cpu().numpy().view(np.uint32).copy())
        if ref is None:
            ref = out
        else:
            np.testing.assert_array_equal(out[0], ref[0])
            np.testing.assert_array_equal(out[1], ref[1])
    assert g.plan.status() == 0


@pytest.mark.parametrize("mode", GRAPH_MODES)
def test_cuda_graph_replay(cases, mode):
    """x + f captured once in a CUDA graph and replayed three times: the fused
    kernels' epochs come from their ever-increasing tickets, so replays (and
    direct calls mixed with them) stay exact."""
    import torch
    w, xyz, dom, o, g = cases("water24k_2x4x8")
    g.plan.set_mode(mode)
    try:
        loc = g.plan.load_home(g.xyz_d)
        f0 = synth.forces(o.n_local_total, seed=4)
        f = torch.from_numpy(f0).cuda()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            g.plan.exchange_x(loc)          # warm-up outside capture, on the capture stream
            g.plan.exchange_f(torch.zeros_like(f))
            with torch.cuda.graph(graph, stream=s):
                g.plan.exchange_x(loc)
                g.plan.exchange_f(f)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        want_x = o.load_home(xyz)
        o.exchange_x(want_x)
        want_f = f0.copy()
        for rep in range(3):
            loc.copy_(g.plan.load_home(g.xyz_d))
            graph.replay()
            o.exchange_f(want_f)
            torch.cuda.synchronize()
            assert g.plan.status() == 0
            np.testing.assert_array_equal(bits(loc.cpu().numpy()), bits(want_x))
            np.testing.assert_array_equal(bits(f.cpu().numpy()), bits(want_f), err_msg="replay %d" % rep)
        # a direct call after the replays still agrees
        g.plan.exchange_f(f)
        o.exchange_f(want_f)
        assert g.plan.status() == 0
        np.testing.assert_array_equal(bits(f.cpu().numpy()), bits(want_f))
    finally:
        g.plan.set_mode("fused")


# -- corner pruning -------------------------------------------------------------------
@pytest.mark.parametrize("name", WORKLOADS)
def test_pruned_plan_and_exchange_parity(name):
    """HALO_SETUP_PRUNE_CORNERS: maps, sizes, shifts and both exchanges in every
    mode bit-identical to the pruning oracle; a rebuild keeps the option."""
    w = synth.WORKLOADS[name]
    xyz, dom = synth.system(w)
    o = oracle.Oracle(w.box, w.grid, w.rc, xyz, dom, prune=True)
    g = gpu_plan(w.box, w.grid, w.rc, xyz, dom, prune=True)
    try:
        assert g.plan.prune
        compare_plans(g, o)
        for mode in MODES:
            g.plan.set_mode(mode)
            compare_exchanges(g, o, xyz, reps=1)
        if name == "water3M_8x8x8":
            xk, dk = synth.displaced(xyz, w.box, w.grid, k=1)
            g.rebuild(xk, dk)
            assert g.plan.prune
            ok = oracle.Oracle(w.box, w.grid, w.rc, xk, dk, prune=True)
            compare_plans(g, ok)
            compare_exchanges(g, ok, xk, reps=1)
    finally:
        g.close()


@pytest.mark.parametrize("box,grid,rc,n,seed", EDGE)
def test_pruned_edge_cases(box, grid, rc, n, seed):
    xyz, dom = synth.custom_system(n, box, grid, seed=seed)
    o = oracle.Oracle(box, grid, rc, xyz, dom, prune=True)
    g = gpu_plan(box, grid, rc, xyz, dom, prune=True)
    try:
        compare_plans(g, o)
        for mode in MODES:
            g.plan.set_mode(mode)
            compare_exchanges(g, o, xyz, reps=1)
    finally:
        g.close()


def test_setup_ex_rejects_unknown_flags():
    import torch
    from domain_decomposition_halo_build_gb300 import halo
    xyz, dom = synth.custom_system(100, (3, 3, 3), (3, 1, 1), seed=1)
    x = torch.from_numpy(xyz).cuda()
    d = torch.from_numpy(dom).cuda()
    with pytest.raises(halo.HaloError) as e:
        halo.halo_setup_ex((3, 3, 3), (3, 1, 1), 0.5, x, d, 2)
    assert e.value.code == halo.EINVAL


@pytest.mark.parametrize("name", ["water24k_2x4x8", "water1M_4x4x4"])
def test_store_home_round_trip_and_forces(cases, name):
    """halo_store_home is the inverse of halo_load_home, and after the force
    reduction it returns every atom's total force in input order: the oracle's
    home slots, placed by their global ids."""
    import torch
    w, xyz, dom, o, g = cases(name)
    loc = g.plan.load_home(g.xyz_d)
    back = g.plan.store_home(loc)
    np.testing.assert_array_equal(bits(back.cpu().numpy()), bits(xyz))
    f0 = synth.forces(o.n_local_total, seed=8)
    want_local = f0.copy()
    o.exchange_f(want_local)
    gid, home, _ = pins.home_slot_of(o)
    want = want_local[home]
    f = torch.from_numpy(f0).cuda()
    g.plan.exchange_f(f)
    got = g.plan.store_home(f)
    assert g.plan.status() == 0
    np.testing.assert_array_equal(bits(got.cpu().numpy()), bits(want))


def random_problem(seed):
    """A seeded random decomposition: grid 1..5 per dim, box 2..8 nm, a cut-off
    that gives 1..(n_d - 1) pulses in decomposed dims, 50..20000 atoms."""
    rng = np.random.default_rng(1000 + seed)
    grid = tuple(int(v) for v in rng.integers(1, 6, size=3))
    box = tuple(float(np.float32(v)) for v in rng.uniform(2.0, 8.0, size=3))
    widths = [box[d] / grid[d] for d in range(3) if grid[d] > 1]
    if widths:
        # the largest rc with p_d = ceil(rc / w_d) <= n_d - 1 in every decomposed dim
        cap = min((grid[d] - 1) * box[d] / grid[d] for d in range(3) if grid[d] > 1)
        rc = float(rng.uniform(0.05, 1.0) * cap * 0.999)
    else:
        rc = float(rng.uniform(0.1, 1.0))
    n = int(rng.integers(50, 20000))
    return box, grid, rc, n, bool(rng.integers(0, 2))


@pytest.mark.parametrize("seed", range(24))
def test_random_problems(seed):
    """Random boxes, grids, cut-offs and sizes, with and without pruning: plans
    and every mode's exchanges bit-identical to the oracle."""
    box, grid, rc, n, prune = random_problem(seed)
    xyz, dom = synth.custom_system(n, box, grid, seed=seed)
    try:
        o = oracle.Oracle(box, grid, rc, xyz, dom, prune=prune)
    except oracle.OracleError as e:
        pytest.skip("oracle rejects the problem (%d)" % e.code)
    g = gpu_plan(box, grid, rc, xyz, dom, prune=prune)
    try:
        compare_plans(g, o)
        for mode in MODES:
            g.plan.set_mode(mode)
            compare_exchanges(g, o, xyz, reps=1, seed=seed)
    finally:
        g.close()


@pytest.mark.parametrize("mode", MODES)
def test_two_plans_on_two_streams(mode):
    """Two independent systems exchanged concurrently on two streams (20
    rounds each, interleaved launches): plans share no device state, so both
    stay bit-identical to the oracle."""
    import torch
    sysA = synth.WORKLOADS["water24k_2x4x8"]
    sysB = synth.WORKLOADS["water48k_2x2x2"]
    runs = []
    for w in (sysA, sysB):
        xyz, dom = synth.system(w)
        o = oracle.Oracle(w.box, w.grid, w.rc, xyz, dom)
        g = gpu_plan(w.box, w.grid, w.rc, xyz, dom)
        g.plan.set_mode(mode)
        want_x = o.load_home(xyz)
        o.exchange_x(want_x)
        f0 = synth.forces(o.n_local_total, seed=12)
        want_f = f0.copy()
        o.exchange_f(want_f)
        runs.append(dict(g=g, want_x=want_x, want_f=want_f, f0=torch.from_numpy(f0).cuda(),
                         stream=torch.cuda.Stream()))
    try:
        for r in runs:
            r["loc"] = r["g"].plan.load_home(r["g"].xyz_d)
        torch.cuda.synchronize()
        for _ in range(20):
            for r in runs:
                with torch.cuda.stream(r["stream"]):
                    r["g"].plan.exchange_x(r["loc"], r["stream"])
                    r["f"] = r["f0"].clone()
                    r["g"].plan.exchange_f(r["f"], r["stream"])
        torch.cuda.synchronize()
        for r in runs:
            assert r["g"].plan.status(r["stream"]) == 0
            np.testing.assert_array_equal(bits(r["loc"].cpu().numpy()), bits(r["want_x"]))
            np.testing.assert_array_equal(bits(r["f"].cpu().numpy()), bits(r["want_f"]))
    finally:
        for r in runs:
            r["g"].close()
