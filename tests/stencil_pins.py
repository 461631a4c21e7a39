"""Pins of the stencil oracle (oracle/stencil.py) against what the page and
the mathematics fix, written so that they also run against a planted-mistake
copy of the oracle (tests/test_stencil_oracle.py)."""
from __future__ import annotations

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
GRIDS = [(1, 1, 4), (2, 1, 4), (1, 3, 8), (3, 1, 4), (2, 2, 4), (2, 4, 8), (3, 2, 12)]


def _matrix(px, py, n, seed):
    rng = np.random.default_rng(seed)
    return rng.random((py * n + 2, px * n + 2)).astype(np.float32)


def load_jacobi_golden():
    rows, key, out = [], None, {}
    for line in open(os.path.join(GOLDEN, "stencil_jacobi_2x2.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line in ("before", "after"):
            key, rows = line, []
        elif line == "end":
            out[key] = np.asarray(rows, np.float32)
        else:
            rows.append([float(v) for v in line.split()])
    return out["before"], out["after"]


def load_exchange_golden():
    g = {"ghost": {}}
    for line in open(os.path.join(GOLDEN, "stencil_exchange_2x2.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        v = line.split()
        if v[0] == "ghost":
            g["ghost"][(int(v[1]), v[2])] = np.asarray([float(x) for x in v[3:]], np.float32)
        else:
            g[v[0]] = int(v[1])
    return g


def ghost_cells(S, field, px, py, n, t, side):
    """The ghost cells of tile t on one side, read through the documented layout."""
    v = np.asarray(field).reshape(py * px, n + 2, S.pitch(n))[t]
    c0 = S.COL0
    return {"north": v[0, c0:c0 + n], "south": v[n + 1, c0:c0 + n],
            "west": v[1:n + 1, c0 - 1], "east": v[1:n + 1, c0 + n]}[side]


def matrix_border_mask(S, px, py, n):
    """True on the ghost cells that hold the fixed border of the matrix."""
    m = np.zeros((py, px, n + 2, S.pitch(n)), bool)
    c0 = S.COL0
    for ty in range(py):
        for tx in range(px):
            if ty == 0:
                m[ty, tx, 0, c0:c0 + n] = True
            if ty == py - 1:
                m[ty, tx, n + 1, c0:c0 + n] = True
            if tx == 0:
                m[ty, tx, 1:n + 1, c0 - 1] = True
            if tx == px - 1:
                m[ty, tx, 1:n + 1, c0 + n] = True
    return m.reshape(-1)


def inner_ghost_mask(S, px, py, n):
    """True on the ghost cells an exchange writes (shared block edges)."""
    m = np.zeros((py, px, n + 2, S.pitch(n)), bool)
    c0 = S.COL0
    m[:, :, 0, c0:c0 + n] = True
    m[:, :, n + 1, c0:c0 + n] = True
    m[:, :, 1:n + 1, c0 - 1] = True
    m[:, :, 1:n + 1, c0 + n] = True
    return m.reshape(-1) & ~matrix_border_mask(S, px, py, n)


def unused_mask(S, px, py, n):
    """True on padding and ghost-ring corners (cells no step reads or writes)."""
    m = np.ones((py, px, n + 2, S.pitch(n)), bool)
    c0 = S.COL0
    m[:, :, 1:n + 1, c0 - 1:c0 + n + 1] = False   # block rows with west/east ghosts
    m[:, :, 0, c0:c0 + n] = False
    m[:, :, n + 1, c0:c0 + n] = False
    return m.reshape(-1)


def check_jacobi_golden(S):
    before, after = load_jacobi_golden()
    np.testing.assert_array_equal(S.jacobi_global(before), after)


def check_fixed_points(S):
    """Discrete harmonic integer fields are fixed points of the sweep, exactly:
    a linear field, and i^2 - j^2 (its five-point Laplacian is 2 - 2 = 0)."""
    i, j = np.mgrid[0:14, 0:11].astype(np.float32)
    for f in (3 * i - 2 * j + 5, i * i - j * j, 7 * j + 1):
        f = f.astype(np.float32)
        np.testing.assert_array_equal(S.jacobi_global(f, steps=3), f)
    # and a non-harmonic field is not (the check is not vacuous)
    g = (i * j).astype(np.float32)
    g[3, 4] += 1
    assert not np.array_equal(S.jacobi_global(g), g)


def check_exchange_golden(S):
    g = load_exchange_golden()
    px, py, n = g["px"], g["py"], g["n"]
    i, j = np.mgrid[0:py * n + 2, 0:px * n + 2]
    a = (100 * i + j).astype(np.float32)
    field = S.to_tiles(a, px, py, n)
    for (t, side), want in g["ghost"].items():
        np.testing.assert_array_equal(ghost_cells(S, field, px, py, n, t, side), want,
                                      err_msg="to_tiles %d %s" % (t, side))
    scrambled = field.copy()
    scrambled[inner_ghost_mask(S, px, py, n)] = -1.0
    ex = S.exchange_tiles(scrambled, px, py, n)
    for (t, side), want in g["ghost"].items():
        np.testing.assert_array_equal(ghost_cells(S, ex, px, py, n, t, side), want,
                                      err_msg="exchange %d %s" % (t, side))


def check_decomposition(S):
    """Sweeping every block from its own tile (after an exchange) gives the
    sweep of the whole matrix; the exchange restores scrambled inner ghosts
    and leaves the border, ghost corners and padding alone; the fused step is a
    sweep followed by an exchange; several fused steps follow several sweeps."""
    for k, (px, py, n) in enumerate(GRIDS):
        a = _matrix(px, py, n, seed=k)
        field = S.to_tiles(a, px, py, n)
        np.testing.assert_array_equal(S.from_tiles(field, px, py, n)[1:-1, 1:-1], a[1:-1, 1:-1])
        want = S.jacobi_global(a)
        got = S.jacobi_tiles(field, field, px, py, n)
        np.testing.assert_array_equal(S.from_tiles(got, px, py, n)[1:-1, 1:-1], want[1:-1, 1:-1],
                                      err_msg=str((px, py, n)))
        inner = inner_ghost_mask(S, px, py, n)
        expect = field.copy()
        expect[unused_mask(S, px, py, n)] = 3.0   # padding and ghost corners: left alone
        scrambled = expect.copy()
        scrambled[inner] = -7.0
        ex = S.exchange_tiles(scrambled, px, py, n)
        np.testing.assert_array_equal(ex, expect, err_msg=str((px, py, n)))
        np.testing.assert_array_equal(S.fused_step(field, field, px, py, n),
                                      S.to_tiles(want, px, py, n), err_msg=str((px, py, n)))
        cur, other = field, field.copy()
        for _ in range(4):
            cur, other = S.fused_step(cur, other, px, py, n), cur
        np.testing.assert_array_equal(cur, S.to_tiles(S.jacobi_global(a, 4), px, py, n))


def run_all(S):
    check_jacobi_golden(S)
    check_fixed_points(S)
    check_exchange_golden(S)
    check_decomposition(S)
