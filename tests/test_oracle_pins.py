"""The CPU oracle against what the pages and the mathematics fix (no GPU).

See tests/pins.py for what each check encodes and where it comes from.
"""
import numpy as np
import pytest

import oracle
import pins
from domain_decomposition_halo_build_gb300 import synth

STRUCT = pins.load_pulse_structure()


def make_oracle(box, grid, rc, xyz, dom, prune=False):
    return oracle.Oracle(box, grid, rc, xyz, dom, prune=prune)


# -- hand-worked golden examples ------------------------------------------------
@pytest.mark.parametrize("name", pins.EXAMPLES)
def test_golden_example(name):
    pins.check_example(make_oracle, pins.load_example(name))


# -- the five workloads: pulse structure, neighbours, maps, geometry -------------
SMALL = ["water3k_2x1x1", "water24k_2x4x8", "water48k_2x2x2"]
LARGE = ["water1M_4x4x4", "water3M_8x8x8"]


@pytest.fixture(scope="module")
def plans():
    cache = {}

    def get(name):
        if name not in cache:
            w = synth.WORKLOADS[name]
            xyz, dom = synth.system(w)
            cache[name] = (w, xyz, dom, oracle.Oracle(w.box, w.grid, w.rc, xyz, dom))
        return cache[name]

    return get


@pytest.mark.parametrize("name", SMALL + LARGE)
def test_pulse_structure(plans, name):
    w, xyz, dom, o = plans(name)
    pins.check_pulse_structure(o, STRUCT[name])


@pytest.mark.parametrize("name", SMALL)
def test_geometric_and_neighbours(plans, name):
    w, xyz, dom, o = plans(name)
    pins.check_geometric(o, xyz, dom)
    pins.check_neighbour_count(o, xyz, dom, STRUCT[name]["neighbours"])


@pytest.mark.parametrize("name", LARGE)
def test_geometric_sampled_domains(plans, name):
    w, xyz, dom, o = plans(name)
    nd = o.n_domains
    pins.check_geometric(o, xyz, dom, domains=[0, nd // 3, nd - 1])


@pytest.mark.parametrize("name", SMALL)
def test_maps_and_exchange_x(plans, name):
    w, xyz, dom, o = plans(name)
    pins.check_maps(o)
    pins.check_load_and_exchange_x(o, xyz)


@pytest.mark.parametrize("name", SMALL + ["water1M_4x4x4"])
def test_forces_integer_conservation_and_closed_form(plans, name):
    w, xyz, dom, o = plans(name)
    pins.check_forces_integer(o)


@pytest.mark.parametrize("name", SMALL)
def test_forces_gaussian_rounding_bound(plans, name):
    w, xyz, dom, o = plans(name)
    pins.check_forces_gaussian(o)


def test_first_dependent_pulse_table(plans):
    """Algorithm 4's dependency table for one pulse per dim (z0: none, y0: z0,
    x0: y0).  y0's entries past depOffset refer only to z0's halo; x0's refer to
    y0's halo -- and, under the reading that x0 also forwards corner atoms that
    arrived in z0, to z0's halo too, which the table alone would leave
    un-awaited."""
    w, xyz, dom, o = plans("water48k_2x2x2")
    # start of the y0 slice in each receiver
    y0_start = {o.pulse(s, 1).recv_domain: o.pulse(s, 1).atom_offset
                for s in range(o.n_domains)}
    seen = {1: set(), 2: set()}
    for s in range(o.n_domains):
        for p in (1, 2):
            info = o.pulse(s, p)
            dep = o.index_map(s, p)[info.split:]
            assert info.split < info.send_size  # every pulse forwards something
            assert np.all(dep >= o.n_home[s])
            for idx in dep:
                seen[p].add("z0" if idx < y0_start[s] else "y0")
    assert seen[1] == {"z0"}
    assert seen[2] == {"z0", "y0"}


# -- brute-force pair coverage on tiny inputs -----------------------------------
TINY = [
    ((3.0, 2.6, 2.2), (3, 2, 2), 0.6, 500),   # 3D, one pulse per dim
    ((4.0, 4.0, 4.0), (1, 2, 5), 1.1, 500),   # y + two z pulses, x undecomposed
    ((3.2, 3.2, 3.2), (4, 1, 1), 1.0, 300),   # two x pulses, 1D
    ((2.4, 2.4, 2.4), (3, 3, 3), 1.0, 400),   # two pulses per dim
]


@pytest.mark.parametrize("box,grid,rc,n", TINY)
def test_pair_coverage_bruteforce(box, grid, rc, n):
    xyz, dom = synth.custom_system(n, box, grid, seed=11)
    o = oracle.Oracle(box, grid, rc, xyz, dom)
    checked = pins.check_pair_coverage(o, xyz, dom)
    assert checked > 50
    pins.check_geometric(o, xyz, dom)
    pins.check_maps(o)
    pins.check_forces_integer(o)


# -- error cases -------------------------------------------------------------------
def test_errors():
    xyz, dom = synth.custom_system(100, (3, 3, 3), (3, 1, 1), seed=1)
    with pytest.raises(oracle.OracleError) as e:
        oracle.Oracle((3, 3, 3), (3, 1, 1), 2.5, xyz, dom)   # p_x = 3 >= n_x
    assert e.value.code == oracle.EPULSES
    bad = dom.copy()
    bad[7] = 3
    with pytest.raises(oracle.OracleError) as e:
        oracle.Oracle((3, 3, 3), (3, 1, 1), 0.5, xyz, bad)
    assert e.value.code == oracle.EDOMAIN
    with pytest.raises(oracle.OracleError) as e:
        oracle.Oracle((3, 3, 3), (3, 1, 1), 0.0, xyz, dom)
    assert e.value.code == oracle.EINVAL


def test_degenerate_cases():
    # one domain: no pulses, exchanges are no-ops
    xyz, dom = synth.custom_system(50, (2, 2, 2), (1, 1, 1), seed=3)
    o = oracle.Oracle((2, 2, 2), (1, 1, 1), 0.5, xyz, dom)
    assert o.n_pulses == 0 and o.n_local_total == 50
    pins.check_forces_integer(o)
    # empty domain and a cut-off so small that almost nothing is sent
    xyz, dom = synth.custom_system(40, (4, 4, 4), (4, 1, 1), seed=4)
    xyz[:, 0] = np.minimum(xyz[:, 0], np.float32(2.9))   # domain 3 stays empty
    dom = synth.assign_domains(xyz, (4, 4, 4), (4, 1, 1))
    o = oracle.Oracle((4, 4, 4), (4, 1, 1), 0.05, xyz, dom)
    assert o.n_home[3] == 0
    pins.check_maps(o)
    pins.check_geometric(o, xyz, dom)
    pins.check_forces_integer(o)


# -- corner pruning (optional plan flag) ------------------------------------------
@pytest.fixture(scope="module")
def pruned():
    cache = {}

    def get(name):
        if name not in cache:
            w = synth.WORKLOADS[name]
            xyz, dom = synth.system(w)
            cache[name] = (w, xyz, dom, oracle.Oracle(w.box, w.grid, w.rc, xyz, dom, prune=True))
        return cache[name]

    return get


@pytest.mark.parametrize("name", SMALL)
def test_pruned_geometric_maps_forces(pruned, name):
    w, xyz, dom, o = pruned(name)
    pins.check_geometric(o, xyz, dom)
    pins.check_maps(o)
    pins.check_load_and_exchange_x(o, xyz)
    pins.check_forces_integer(o)


@pytest.mark.parametrize("name", LARGE)
def test_pruned_geometric_sampled_domains(pruned, name):
    w, xyz, dom, o = pruned(name)
    nd = o.n_domains
    pins.check_geometric(o, xyz, dom, domains=[0, nd // 3, nd - 1])


@pytest.mark.parametrize("name", SMALL)
def test_pruned_halo_is_a_subset(plans, pruned, name):
    """Pruning only removes halo images: every domain's pruned set is contained
    in its unpruned set, and on these 3D workloads it removes some."""
    w, xyz, dom, o = plans(name)
    _, _, _, q = pruned(name)
    full, part = pins.halo_images(o, xyz), pins.halo_images(q, xyz)
    removed = 0
    for D in range(o.n_domains):
        assert set(part[D]) <= set(full[D]), D
        removed += len(full[D]) - len(part[D])
    assert (removed > 0) == (int(np.sum(np.asarray(w.grid) > 1)) > 1), removed


def test_pruned_example_prunes_one_atom_that_the_slabs_keep():
    """The hand-worked pruning example built without pruning: the x pulse of
    sender 3 also sends the atom whose corner distance is 1.27 > rc."""
    ex = pins.load_example("tiny_2x2x1_corner_pruned.txt")
    o = oracle.Oracle(ex["box"], ex["grid"], ex["rc"], ex["atoms"], ex["domains"].astype(np.int32))
    np.testing.assert_array_equal(o.index_map(3, 1), [0, 1, 2])


@pytest.mark.parametrize("box,grid,rc,n", TINY)
def test_pruned_pair_coverage_bruteforce(box, grid, rc, n):
    xyz, dom = synth.custom_system(n, box, grid, seed=11)
    o = oracle.Oracle(box, grid, rc, xyz, dom, prune=True)
    assert pins.check_pair_coverage(o, xyz, dom) > 50
    pins.check_geometric(o, xyz, dom)
    pins.check_forces_integer(o)


@pytest.mark.parametrize("name", ["water24k_2x4x8", "water48k_2x2x2"])
def test_threaded_exchanges_match_sequential(plans, name):
    """The senders of one pulse are independent, so the host-threaded exchanges
    (used only to time the oracle on all cores) give the same bits."""
    w, xyz, dom, o = plans(name)
    if not o.openmp:
        pytest.skip("oracle built without OpenMP")
    loc = o.load_home(xyz)
    f = synth.forces(o.n_local_total, seed=5)
    seq_x, seq_f = loc.copy(), f.copy()
    o.exchange_x(seq_x)
    o.exchange_f(seq_f)
    try:
        o.set_threads(4)
        par_x, par_f = loc.copy(), f.copy()
        o.exchange_x(par_x)
        o.exchange_f(par_f)
    finally:
        o.set_threads(1)
    np.testing.assert_array_equal(par_x.view(np.uint32), seq_x.view(np.uint32))
    np.testing.assert_array_equal(par_f.view(np.uint32), seq_f.view(np.uint32))
