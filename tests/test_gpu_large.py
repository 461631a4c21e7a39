"""The library at its largest sizes, checked by properties that hold at any size.

Two 40M-atom systems (about 100 atoms/nm^3, rc 1.2 nm) on either side of the
FLAT mode's limit of 2^26 local slots (home plus halo):
- 8x8x8 domains, about 58M local slots: every mode runs, and FLAT and FUSED
  agree bit for bit;
- 16x16x16 domains, about 80M local slots: FLAT is refused with
  HALO_ECAPACITY, and the plan keeps working in FUSED mode.

The oracle is too slow at these sizes, so the checks are closed forms from
the page "Redesigning GROMACS Halo Exchange: Improving Strong Scaling with
GPU-initiated NVSHMEM" (section 3, the eighth-shell halo; Algorithms 4 and 6):
- every home slot holds its atom's coordinate and lies in its domain's cell;
- every halo slot holds its owner's coordinate, shifted by +L_d (one fp32
  add) in exactly the dims where that puts it into the receiving domain's
  cell widened by rc on its upper side;
- with small integer forces (all sums exact in fp32), every owner's reduced
  force equals its own plus the forces of all its halo copies.
"""
import numpy as np
import pytest

from domain_decomposition_halo_build_gb300 import synth

pytestmark = pytest.mark.gpu

FLAT_SLOT_LIMIT = 1 << 26
RC = 1.2
BOX = 73.7  # 40M atoms at ~100 atoms/nm^3


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def make_plan(grid, seed):
    import torch
    from domain_decomposition_halo_build_gb300 import halo
    box = (BOX, BOX, BOX)
    xyz, dom = synth.custom_system(40_000_000, box, (grid,) * 3, seed=seed)
    x = torch.from_numpy(xyz).cuda()
    d = torch.from_numpy(dom).cuda()
    return halo.HaloPlan(box, (grid,) * 3, RC, x, d), x


def check_coordinates(plan, x, loc):
    """Home slots: the atom's own coordinate, inside its cell.  Halo slots: the
    owner's coordinate plus fl32(+L_d) exactly where the eighth-shell region
    of the receiving domain requires it.  Cell faces are c * L / n in double
    from the fp32 box, as the domain ids are; rc is the fp32 cutoff."""
    import torch
    dev = loc.device
    g = plan_grid(plan)
    l2g = plan.local_to_global().long()
    L32 = torch.tensor([BOX] * 3, dtype=torch.float32, device=dev)
    L64 = L32.double()
    rc = float(np.float32(RC))
    n_local = torch.from_numpy(plan.n_local.astype(np.int64)).to(dev)
    n_home = torch.from_numpy(plan.n_home.astype(np.int64)).to(dev)
    dom_of_slot = torch.repeat_interleave(torch.arange(plan.n_domains, device=dev), n_local)
    base = torch.from_numpy(plan.base).to(dev)
    is_home = torch.arange(plan.n_local_total, device=dev) - base[dom_of_slot] < n_home[dom_of_slot]
    cell = torch.stack([dom_of_slot % g, (dom_of_slot // g) % g, dom_of_slot // (g * g)], 1).double()
    lo = cell * L64 / g
    hi = (cell + 1) * L64 / g
    owner = x[l2g]
    shifted = owner + L32  # one fp32 add per component
    c64 = loc.double()
    # home slots: unchanged, inside the cell
    assert torch.equal(loc[is_home], owner[is_home])
    assert bool(((c64[is_home] >= lo[is_home]) & (c64[is_home] < hi[is_home])).all())
    # halo slots: owner or owner + L per component, inside [lo, hi + rc)
    # (a shifted value may round up by half an fp32 ulp past hi + rc)
    h = ~is_home
    same = loc[h] == owner[h]
    plus = loc[h] == shifted[h]
    assert bool((same | plus).all()), "a halo coordinate is neither its owner's nor owner + L"
    inside = (c64[h] >= lo[h]) & (c64[h] < hi[h] + rc + 1e-5)
    assert bool(inside.all()), "a halo slot lies outside the receiving domain's eighth-shell region"
    # the shift is applied exactly where the unshifted owner lies outside it
    o64 = owner[h].double()
    unshifted_inside = (o64 >= lo[h]) & (o64 < hi[h] + rc)
    assert bool(((plus & ~same) == ~unshifted_inside).all()), "wrong periodic shift"
    return l2g, is_home


def plan_grid(plan):
    return int(round(plan.n_domains ** (1.0 / 3.0)))


def check_forces(plan, f0, f, l2g, is_home):
    """Integer-valued forces: owner result = own force + sum over its copies."""
    import torch
    n_atoms = plan.n_atoms
    want = torch.zeros((n_atoms, 3), dtype=torch.float64, device=f.device)
    want.index_add_(0, l2g, f0.double())  # own slot plus every copy, exact in fp64
    got = torch.empty_like(want)
    got[l2g[is_home]] = f[is_home].double()
    assert torch.equal(got, want)


def run_mode(plan, x, mode, seed=5):
    import torch
    plan.set_mode(mode)
    loc = plan.load_home(x)
    plan.exchange_x(loc)
    gen = torch.Generator(device="cuda").manual_seed(seed)
    f0 = torch.randint(-8, 9, (plan.n_local_total, 3), generator=gen, device="cuda").float()
    f = f0.clone()
    plan.exchange_f(f)
    assert plan.status() == 0
    return loc, f0, f


def test_largest_flat_plan_matches_fused_and_closed_forms():
    import torch
    plan, x = make_plan(8, seed=11)
    try:
        assert plan.n_local_total < FLAT_SLOT_LIMIT
        assert plan.n_local_total > (FLAT_SLOT_LIMIT * 3) // 4, plan.n_local_total
        loc_flat, f0, f_flat = run_mode(plan, x, "flat")
        l2g, is_home = check_coordinates(plan, x, loc_flat)
        check_forces(plan, f0, f_flat, l2g, is_home)
        loc_fused, f0b, f_fused = run_mode(plan, x, "fused")
        assert torch.equal(f0, f0b)
        # the same bits in both modes (the chained and the composed exchange)
        assert torch.equal(loc_fused.view(torch.int32), loc_flat.view(torch.int32))
        assert torch.equal(f_fused.view(torch.int32), f_flat.view(torch.int32))
    finally:
        plan.close()


def test_beyond_the_flat_limit_fused_still_exact():
    from domain_decomposition_halo_build_gb300 import halo
    plan, x = make_plan(16, seed=12)
    try:
        assert plan.n_local_total >= FLAT_SLOT_LIMIT, plan.n_local_total
        with pytest.raises(halo.HaloError) as e:
            plan.set_mode("flat")
        assert e.value.code == halo.ECAPACITY
        assert plan.mode == "fused"
        loc, f0, f = run_mode(plan, x, "fused")
        l2g, is_home = check_coordinates(plan, x, loc)
        check_forces(plan, f0, f, l2g, is_home)
    finally:
        plan.close()
