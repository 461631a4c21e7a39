"""CPU oracle for the two-dimensional stencil halo workload -- TEST INFRASTRUCTURE.

Written from the page "GPU-centric Communication on NVIDIA GPU Clusters with
InfiniBand: A Case Study with OpenSHMEM", section "2D stencil mini-app":
  - data partitioning: every rank holds one square block of the matrix; the
    ranks form a one- or two-dimensional grid that is not periodic (a corner
    rank talks to two neighbours, an edge rank to three, an interior rank to
    four);
  - every iteration a rank computes its block and sends its boundary to its
    neighbours; the received boundary is used by the next iteration's kernel
    (the kernel boundary gives the consistency);
  - the MPI version runs separate kernels for computing and packing, the
    GPU-initiated version one fused kernel that computes and sends.
Readings where the page is silent (each one is also listed in the design
notes): the stencil is the five-point Jacobi sweep with weight 1/4 in fp32,
evaluated as ((N + S) + (W + E)) * 0.25; the cells around the whole matrix hold
fixed (Dirichlet) values that no step changes; a block exchanges its edge rows
and columns only (the five-point stencil never reads a diagonal neighbour).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may
import this module; the library never does.  numpy float32 arithmetic is
IEEE single precision with one rounding per operation.

Tile layout (the library's, described here so that whole buffers compare):
tiles are stored one after another, tile t = tx + px * ty (tx along the
columns, ty along the rows), each (n + 2) rows of pitch(n) = n + 8 floats:
row 0 is the ghost row above the block, rows 1..n the block, row n + 1 the
ghost row below; columns 4..n+3 are the block (16-byte aligned), column 3 the
west ghost, column n + 4 the east ghost, the rest padding.

The global matrix is an (py*n + 2) x (px*n + 2) float32 array whose outer ring
is the fixed border; block (tx, ty) is rows 1 + ty*n .. ty*n + n and columns
1 + tx*n .. tx*n + n.
"""
from __future__ import annotations

import numpy as np

COL0 = 4  # first block column inside a tile row


def pitch(n: int) -> int:
    return n + 8


def tile_floats(n: int) -> int:
    return (n + 2) * pitch(n)


def jacobi_global(a: np.ndarray, steps: int = 1) -> np.ndarray:
    """`steps` five-point Jacobi sweeps of the whole matrix (border fixed)."""
    a = np.array(a, dtype=np.float32, copy=True)
    q = np.float32(0.25)
    for _ in range(steps):
        b = a.copy()
        ns = a[:-2, 1:-1] + a[2:, 1:-1]
        we = a[1:-1, :-2] + a[1:-1, 2:]
        b[1:-1, 1:-1] = (ns + we) * q
        a = b
    return a


def _view(field: np.ndarray, px: int, py: int, n: int) -> np.ndarray:
    return field.reshape(py, px, n + 2, pitch(n))


def to_tiles(a: np.ndarray, px: int, py: int, n: int) -> np.ndarray:
    """The tile field of matrix `a` after a completed exchange: every block,
    and around it the cells its stencil reads (the neighbouring blocks' edge
    cells, or the fixed border).  Padding and ghost-ring corners are 0."""
    a = np.asarray(a, np.float32)
    assert a.shape == (py * n + 2, px * n + 2)
    out = np.zeros((py, px, n + 2, pitch(n)), np.float32)
    for ty in range(py):
        for tx in range(px):
            blk = a[ty * n:ty * n + n + 2, tx * n:tx * n + n + 2]
            t = out[ty, tx]
            t[1:n + 1, COL0:COL0 + n] = blk[1:n + 1, 1:n + 1]
            t[0, COL0:COL0 + n] = blk[0, 1:n + 1]
            t[n + 1, COL0:COL0 + n] = blk[n + 1, 1:n + 1]
            t[1:n + 1, COL0 - 1] = blk[1:n + 1, 0]
            t[1:n + 1, COL0 + n] = blk[1:n + 1, n + 1]
    return out.reshape(-1)


def from_tiles(field: np.ndarray, px: int, py: int, n: int) -> np.ndarray:
    """The matrix held by a tile field: blocks, and the border from the ghost
    cells of the blocks on the matrix edge (the four corner cells are 0)."""
    v = _view(np.asarray(field, np.float32), px, py, n)
    a = np.zeros((py * n + 2, px * n + 2), np.float32)
    for ty in range(py):
        for tx in range(px):
            t = v[ty, tx]
            r, c = 1 + ty * n, 1 + tx * n
            a[r:r + n, c:c + n] = t[1:n + 1, COL0:COL0 + n]
            if ty == 0:
                a[0, c:c + n] = t[0, COL0:COL0 + n]
            if ty == py - 1:
                a[r + n, c:c + n] = t[n + 1, COL0:COL0 + n]
            if tx == 0:
                a[r:r + n, 0] = t[1:n + 1, COL0 - 1]
            if tx == px - 1:
                a[r:r + n, c + n] = t[1:n + 1, COL0 + n]
    return a


def exchange_tiles(field: np.ndarray, px: int, py: int, n: int) -> np.ndarray:
    """One halo exchange: each block's first and last rows go to the ghost
    rows of the blocks above and below it, its first and last columns to the
    ghost columns of the blocks left and right of it.  Ghost cells on the
    matrix border, ghost-ring corners and padding are left as they are."""
    out = np.array(field, dtype=np.float32, copy=True)
    src = _view(np.asarray(field, np.float32), px, py, n)
    dst = _view(out, px, py, n)
    for ty in range(py):
        for tx in range(px):
            t = src[ty, tx]
            if ty > 0:       # block above receives my first row below its block
                dst[ty - 1, tx][n + 1, COL0:COL0 + n] = t[1, COL0:COL0 + n]
            if ty < py - 1:  # block below receives my last row above its block
                dst[ty + 1, tx][0, COL0:COL0 + n] = t[n, COL0:COL0 + n]
            if tx > 0:       # block on the left receives my first column
                dst[ty, tx - 1][1:n + 1, COL0 + n] = t[1:n + 1, COL0]
            if tx < px - 1:  # block on the right receives my last column
                dst[ty, tx + 1][1:n + 1, COL0 - 1] = t[1:n + 1, COL0 + n - 1]
    return out


def jacobi_tiles(field_in: np.ndarray, field_out: np.ndarray, px: int, py: int,
                 n: int) -> np.ndarray:
    """One Jacobi sweep of every block from its own tile alone (block and ghost
    cells of `field_in`); returns `field_out` with the blocks replaced and
    everything else as it was."""
    src = _view(np.asarray(field_in, np.float32), px, py, n)
    out = np.array(field_out, dtype=np.float32, copy=True)
    dst = _view(out, px, py, n)
    q = np.float32(0.25)
    for ty in range(py):
        for tx in range(px):
            t = src[ty, tx]
            ns = t[0:n, COL0:COL0 + n] + t[2:n + 2, COL0:COL0 + n]
            we = t[1:n + 1, COL0 - 1:COL0 + n - 1] + t[1:n + 1, COL0 + 1:COL0 + n + 1]
            dst[ty, tx][1:n + 1, COL0:COL0 + n] = (ns + we) * q
    return out


def fused_step(field_in: np.ndarray, field_out: np.ndarray, px: int, py: int,
               n: int) -> np.ndarray:
    """The fused iteration (the page's single kernel that computes and sends):
    a sweep of every block followed by the exchange of the new values."""
    return exchange_tiles(jacobi_tiles(field_in, field_out, px, py, n), px, py, n)
