"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix, independent of the oracle's own code.

Sources (page "Redesigning GROMACS Halo Exchange: Improving Strong Scaling with
GPU-initiated NVSHMEM", review):
  * section 3: each domain owns its home atoms; atoms within the cut-off of a
    face are forwarded through intermediate domains (eighth shell), phases
    z -> y -> x, reaching np(x)np(y)np(z) - 1 neighbours in np(x)+np(y)+np(z)
    pulses;
  * Algorithm 1 (PulseData), Algorithm 4 (depOffset split, global pulse order
    Z -> Y -> X, firstDependentPulse), Algorithm 6 (forces back to owners,
    last pulse first).

Each check raises AssertionError with a message on the first violation.
"""
from __future__ import annotations

import os
from collections import defaultdict

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# --------------------------------------------------------------------------- #
# golden fixtures
# --------------------------------------------------------------------------- #
def load_pulse_structure():
    rows = {}
    with open(os.path.join(GOLDEN, "pulse_structure.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, px, py, pz, P, order, nb = line.split()
            rows[name] = dict(per_dim=(int(px), int(py), int(pz)), P=int(P),
                              order=order.split(","), neighbours=int(nb))
    return rows


def load_example(name):
    """Parse one hand-worked example under tests/golden/."""
    ex = {"pulses": {}}
    with open(os.path.join(GOLDEN, name)) as f:
        lines = [ln.strip() for ln in f]
    i = 0
    while i < len(lines):
        ln = lines[i]
        i += 1
        if not ln or ln.startswith("#"):
            continue
        key, _, rest = ln.partition(" ")
        if key in ("atoms", "local_coords", "forces_before", "forces_after"):
            rows = []
            while lines[i] != "end":
                rows.append([float(v) for v in lines[i].split()])
                i += 1
            i += 1
            ex[key] = np.asarray(rows, dtype=np.float32)
        elif key == "pulse":
            head, _, mp = rest.partition(":")
            v = head.split()
            s, p = int(v[0]), int(v[1])
            ex["pulses"][(s, p)] = dict(
                recv_domain=int(v[2]), send_size=int(v[3]), split=int(v[4]),
                dep_offset=int(v[5]), atom_offset=int(v[6]),
                shift=np.asarray([float(x) for x in v[7:10]], np.float32),
                map=np.asarray([int(x) for x in mp.split()], np.int32))
        elif key in ("box",):
            ex[key] = np.asarray([float(x) for x in rest.split()], np.float32)
        elif key == "rc":
            ex[key] = float(rest)
        else:
            ex[key] = np.asarray([int(x) for x in rest.split()], np.int64)
    return ex


EXAMPLES = ["tiny_2x1x1.txt", "tiny_4x1x1_two_pulse.txt", "tiny_2x2x1_corner.txt",
            "tiny_2x2x1_corner_pruned.txt"]


def check_example(make_plan, ex):
    """Compare a plan (oracle or library adaptor) with a hand-worked example.

    ``make_plan(box, grid, rc, xyz, dom, prune=...)`` returns an object with
    the attributes/methods of ``oracle.Oracle``.
    """
    prune = bool(ex["prune"][0]) if "prune" in ex else False
    o = make_plan(ex["box"], ex["grid"], ex["rc"], ex["atoms"], ex["domains"].astype(np.int32),
                  prune=prune)
    assert list(o.pulse_dim) == list(ex["pulse_dims"]), ("pulse dims", o.pulse_dim)
    np.testing.assert_array_equal(o.n_home, ex["n_home"], err_msg="n_home")
    np.testing.assert_array_equal(o.n_local, ex["n_local"], err_msg="n_local")
    np.testing.assert_array_equal(o.base, ex["base"], err_msg="base")
    for (s, p), want in ex["pulses"].items():
        got = o.pulse(s, p)
        for k in ("recv_domain", "send_size", "split", "dep_offset", "atom_offset"):
            assert getattr(got, k) == want[k], ((s, p), k, getattr(got, k), want[k])
        np.testing.assert_array_equal(got.coord_shift, want["shift"], err_msg=str((s, p)))
        np.testing.assert_array_equal(o.index_map(s, p), want["map"], err_msg=str((s, p)))
    np.testing.assert_array_equal(o.local_to_global(), ex["local_to_global"])
    loc = o.load_home(ex["atoms"])
    o.exchange_x(loc)
    np.testing.assert_array_equal(loc, ex["local_coords"], err_msg="local coords")
    f = ex["forces_before"].copy()
    o.exchange_f(f)
    np.testing.assert_array_equal(f, ex["forces_after"], err_msg="forces after")


# --------------------------------------------------------------------------- #
# structural checks
# --------------------------------------------------------------------------- #
def cells_of(dom, grid):
    dom = np.asarray(dom, np.int64)
    nx, ny = int(grid[0]), int(grid[1])
    return np.stack([dom % nx, (dom // nx) % ny, dom // (nx * ny)], axis=1)


def check_pulse_structure(o, expect):
    """Pulse counts and the z -> y -> x order against the hand-derived table."""
    assert tuple(int(v) for v in o.pulses_per_dim) == expect["per_dim"], o.pulses_per_dim
    assert o.n_pulses == expect["P"] == sum(expect["per_dim"])
    names = []
    count = defaultdict(int)
    for d in o.pulse_dim:
        names.append("xyz"[d] + str(count[d]))
        count[d] += 1
    assert names == expect["order"], names


def halo_images(o, xyz):
    """For every domain, the multiset of (owner gid, image shift in box
    lengths per component) of its halo slots, read from the plan's local
    coordinates.  A slot whose coordinate is neither the owner's nor the owner's
    plus one box length in a component is reported with shift code 9."""
    gid = o.local_to_global()
    loc = o.local_coords() if hasattr(o, "local_coords") else None
    L = np.asarray(o.box, np.float32)
    out = {}
    for D in range(o.n_domains):
        lo = int(o.base[D]) + int(o.n_home[D])
        hi = int(o.base[D]) + int(o.n_local[D])
        g = gid[lo:hi]
        c = loc[lo:hi]
        own = xyz[g]
        code = np.full(c.shape, 9, np.int64)
        code[c == own] = 0
        code[c == (own + L[None, :]).astype(np.float32)] = 1
        out[D] = sorted(zip(g.tolist(), *[code[:, e].tolist() for e in range(3)]))
    return out


def geometric_halo(xyz, dom, box, grid, rc, per_dim, domains=None, prune=False):
    """Direct construction of every domain's eighth-shell halo, atom by atom.

    An atom whose home cell is H appears in domain D's halo iff, in every
    decomposed dim d, its cell offset o_d = (H_d - D_d) mod n_d is in [0, p_d],
    not all offsets are zero, and for every forwarding step j = o_d ... 1 the
    coordinate, as held by the domain at offset j, lies below that domain's
    lower face plus the cut-off (fp32 threshold fl32(S*L/n + rc)).  The
    coordinate held at offset j carries +L_d iff the chain crossed the
    periodic boundary between offset o_d and offset j.  Image shift = +L_d iff
    D_d + o_d >= n_d.

    prune (corner pruning): at every forwarding step the atom must also lie
    within rc of the receiving domain's box over the dims in which it is beyond
    that box.  Steps go z, then y, then x; at step j of dim d the receiving
    domain is at offset j - 1 in d and already at D in the dims forwarded
    before d, so the distance is
        max(0, held_d - lower face of the domain at offset j)^2
      + sum over earlier-forwarded dims e with o_e > 0, ascending e, of
        max(0, x_e as held in D - upper face of D in e)^2
    in double, compared with rc^2 (rc as fp32, squared in double).
    """
    L = np.asarray(box, np.float32)
    n = np.asarray(grid, np.int64)
    cells = cells_of(dom, grid)
    N = xyz.shape[0]
    nd = int(np.prod(n))
    rc2 = float(np.float32(rc)) * float(np.float32(rc))
    out = {}
    for D in (range(nd) if domains is None else domains):
        cD = cells_of(np.asarray([D]), grid)[0]
        ok = np.ones(N, bool)
        moved = np.zeros(N, bool)
        shift = np.zeros((N, 3), np.int64)
        final = {}   # dim -> (offset, coordinate as held in D)
        for d in (2, 1, 0):
            if n[d] == 1:
                continue
            o = (cells[:, d] - cD[d]) % n[d]
            ok &= o <= per_dim[d]
            wrap_o = (cD[d] + o) >= n[d]
            x = xyz[:, d]
            xs = (x + L[d]).astype(np.float32)
            for j in range(1, int(per_dim[d]) + 1):
                U = cD[d] + j
                S = U % n[d]
                held = np.where(wrap_o & (U < n[d]), xs, x)
                thr = np.float32(float(S) * float(L[d]) / float(n[d]) + float(np.float32(rc)))
                step_ok = held < thr
                if prune:
                    lo = float(S) * float(L[d]) / float(n[d])
                    t = np.maximum(held.astype(np.float64) - lo, 0.0)
                    r2 = t * t
                    for e in (0, 1, 2):
                        if e == d or e not in final:
                            continue
                        oe, xe = final[e]
                        hi = float(cD[e] + 1) * float(L[e]) / float(n[e])
                        u = np.maximum(xe.astype(np.float64) - hi, 0.0)
                        r2 = r2 + np.where(oe > 0, u * u, 0.0)
                    step_ok &= r2 < rc2
                ok &= (o < j) | step_ok
            shift[:, d] = wrap_o.astype(np.int64)
            moved |= o > 0
            final[d] = (o, np.where(wrap_o, xs, x))
        ok &= moved
        idx = np.nonzero(ok)[0]
        out[D] = sorted(zip(idx.tolist(), *[shift[idx, e].tolist() for e in range(3)]))
    return out


def check_geometric(o, xyz, dom, domains=None):
    per_dim = [int(v) for v in o.pulses_per_dim]
    want = geometric_halo(xyz, dom, o.box, o.grid, o.rc, per_dim, domains,
                          prune=getattr(o, "prune", False))
    got = halo_images(o, xyz)
    for D, w in want.items():
        g = got[D]
        assert len(set(g)) == len(g), ("duplicate halo image", D)
        assert g == w, ("halo set of domain", D, len(g), len(w),
                        sorted(set(g) ^ set(w))[:5])


def check_neighbour_count(o, xyz, dom, expect_neighbours):
    """Distinct (home domain, image) sources in each domain's halo =
    prod(p_d + 1) - 1 (page: np(x)np(y)np(z) - 1 neighbours, zone-count
    reading)."""
    gid = o.local_to_global()
    dom = np.asarray(dom)
    imgs = halo_images(o, xyz)
    for D in range(o.n_domains):
        src = {(int(dom[g]), sx, sy, sz) for g, sx, sy, sz in imgs[D]}
        assert len(src) == expect_neighbours, (D, len(src), expect_neighbours)
    return gid


def check_maps(o):
    """Index-map invariants: ascending unique entries drawn from the pulse's
    candidate range; split = entries below depOffset = n_home; entries past
    depOffset refer to halo slots received in earlier pulses; receiver is
    s - e_d; each receiver's pulse slices tile its local range in order;
    coordShift is +L_d exactly when s_d == 0."""
    P = o.n_pulses
    grid = np.asarray(o.grid)
    L = np.asarray(o.box, np.float32)
    recv_slices = defaultdict(list)
    starts = {}
    for p in range(P):
        d = int(o.pulse_dim[p])
        for s in range(o.n_domains):
            info = o.pulse(s, p)
            m = o.index_map(s, p)
            c = cells_of(np.asarray([s]), grid)[0]
            rc_ = c.copy()
            rc_[d] = (c[d] - 1) % grid[d]
            r = int(rc_[0] + grid[0] * (rc_[1] + grid[1] * rc_[2]))
            assert info.recv_domain == r, ("receiver", s, p)
            assert info.send_size == len(m)
            assert np.all(np.diff(m) > 0), ("map not ascending/unique", s, p)
            assert info.dep_offset == o.n_home[s]
            assert info.split == int(np.sum(m < o.n_home[s])), ("split", s, p)
            want_shift = np.zeros(3, np.float32)
            if c[d] == 0:
                want_shift[d] = L[d]
            np.testing.assert_array_equal(info.coord_shift, want_shift)
            if len(m):
                assert m[0] >= 0
            recv_slices[r].append((p, info.atom_offset, info.send_size))
            starts[(r, p)] = info.atom_offset
    for r, sl in recv_slices.items():
        sl.sort()
        pos = int(o.n_home[r])
        for p, off, n in sl:
            assert off == pos, ("slice start", r, p, off, pos)
            pos += n
        assert pos == o.n_local[r]
    # candidate ranges
    for p in range(P):
        d = int(o.pulse_dim[p])
        first_of_dim = p == 0 or int(o.pulse_dim[p - 1]) != d
        for s in range(o.n_domains):
            m = o.index_map(s, p)
            if not len(m):
                continue
            assert m[-1] < starts[(s, p)], ("entry beyond candidates", s, p)
            if not first_of_dim:
                assert m[0] >= starts[(s, p - 1)], ("forwarded pulse reaches back", s, p)


def check_load_and_exchange_x(o, xyz):
    """Home slots hold the owners' coordinates; exchange_x reproduces the
    build-time halo exactly."""
    gid = o.local_to_global()
    built = o.local_coords()
    loc = o.load_home(xyz)
    for D in range(o.n_domains):
        b, h = int(o.base[D]), int(o.n_home[D])
        np.testing.assert_array_equal(loc[b:b + h], xyz[gid[b:b + h]])
    o.exchange_x(loc)
    np.testing.assert_array_equal(loc, built, err_msg="exchange_x != build-time fill")


def home_slot_of(o):
    gid = o.local_to_global()
    home = np.full(o.n_atoms, -1, np.int64)
    is_home = np.zeros(o.n_local_total, bool)
    for D in range(o.n_domains):
        b, h = int(o.base[D]), int(o.n_home[D])
        home[gid[b:b + h]] = np.arange(b, b + h)
        is_home[b:b + h] = True
    assert np.all(home >= 0)
    return gid, home, is_home


def check_forces_integer(o, seed=5):
    """Integer-valued forces: total force conserved exactly and each owner
    receives exactly its own force plus the forces of all its halo copies."""
    rng = np.random.default_rng(seed)
    f0 = rng.integers(-8, 9, size=(o.n_local_total, 3)).astype(np.float32)
    f = f0.copy()
    o.exchange_f(f)
    gid, home, is_home = home_slot_of(o)
    tot_before = f0.astype(np.float64).sum(axis=0)
    tot_after = f[is_home].astype(np.float64).sum(axis=0)
    np.testing.assert_array_equal(tot_after, tot_before, err_msg="force not conserved")
    want = np.zeros((o.n_atoms, 3), np.float64)
    np.add.at(want, gid, f0.astype(np.float64))
    np.testing.assert_array_equal(f[home].astype(np.float64), want,
                                  err_msg="owner force != sum of copies")


def check_forces_gaussian(o, seed=6):
    """N(0,1) forces: owner force = own + sum of copies within fp32 rounding of
    the k adds (k = number of copies)."""
    rng = np.random.default_rng(seed)
    f0 = rng.standard_normal((o.n_local_total, 3)).astype(np.float32)
    f = f0.copy()
    o.exchange_f(f)
    gid, home, _ = home_slot_of(o)
    want = np.zeros((o.n_atoms, 3), np.float64)
    absum = np.zeros((o.n_atoms, 3), np.float64)
    np.add.at(want, gid, f0.astype(np.float64))
    np.add.at(absum, gid, np.abs(f0.astype(np.float64)))
    copies = np.bincount(gid, minlength=o.n_atoms)[:, None].astype(np.float64)
    tol = copies * 2.0 ** -24 * absum + 1e-30
    err = np.abs(f[home].astype(np.float64) - want)
    assert np.all(err <= tol), ("rounding bound exceeded", float(np.max(err / tol)))


def check_pair_coverage(o, xyz, dom, margin=1e-4):
    """Brute force on a tiny input: every pair of atoms in different domains
    closer than rc (minimum image) is co-present in some domain, at local
    separation equal to the minimum-image separation (undecomposed dims are
    compared modulo the box)."""
    L = np.asarray(o.box, np.float64)
    grid = np.asarray(o.grid)
    rc = float(o.rc)
    gid = o.local_to_global()
    loc = o.local_coords().astype(np.float64)
    holders = defaultdict(list)
    for D in range(o.n_domains):
        b, n = int(o.base[D]), int(o.n_local[D])
        for j in range(b, b + n):
            holders[int(gid[j])].append((D, j))
    x = xyz.astype(np.float64)
    dom = np.asarray(dom)
    N = x.shape[0]
    checked = 0
    for a in range(N):
        dv = x[a + 1:] - x[a]
        dv -= L * np.round(dv / L)
        dist = np.sqrt((dv ** 2).sum(axis=1))
        for k in np.nonzero((dist < rc * (1 - margin)) & (dom[a + 1:] != dom[a]))[0]:
            b = a + 1 + int(k)
            want = dv[k]
            ha = defaultdict(list)
            for D, j in holders[a]:
                ha[D].append(j)
            found = False
            for D, jb in holders[b]:
                for ja in ha.get(D, ()):
                    sep = loc[jb] - loc[ja]
                    for d in range(3):
                        if grid[d] == 1:
                            sep[d] -= L[d] * np.round(sep[d] / L[d])
                    if np.all(np.abs(sep - want) < 1e-4):
                        found = True
                        break
                if found:
                    break
            assert found, ("pair not co-present", a, b, float(dist[k]))
            checked += 1
    return checked
