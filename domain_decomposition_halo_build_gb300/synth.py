"""Seeded synthetic inputs for the halo exchange.

This module holds only random draws: atom positions, the domain id of each
atom (the cell its position falls in), halo forces and the per-rebuild
displacements.  It holds none of the exchange's arithmetic, so both the CUDA
path and the CPU oracle consume its output.

The systems stand in for the water-ethanol benchmark systems of the page
"Redesigning GROMACS Halo Exchange: Improving Strong Scaling with
GPU-initiated NVSHMEM" (section 6, benchmark systems), which are not
available here: atoms are uniform-random in a cubic periodic box at about
100 atoms/nm^3, roughly the density of liquid water.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    n_atoms: int
    box: tuple
    grid: tuple
    rc: float
    seed: int = 0
    rebuild_every: int = 0  # exchanges between rebuilds (0: never)
    description: str = ""


WORKLOADS = {
    w.name: w
    for w in (
        Workload("water3k_2x1x1", 3000, (3.1, 3.1, 3.1), (2, 1, 1), 1.0,
                 description="3,000 atoms, 3.1 nm box, 2x1x1 domains, rc 1.0 nm, 1 pulse in x"),
        Workload("water24k_2x4x8", 24000, (6.2, 6.2, 6.2), (2, 4, 8), 1.2,
                 description="24,000 atoms, 6.2 nm box, 2x4x8 domains, rc 1.2 nm, "
                             "2 z-pulses + 1 y + 1 x"),
        Workload("water48k_2x2x2", 48000, (7.8, 7.8, 7.8), (2, 2, 2), 1.0,
                 description="48,000 atoms, 7.8 nm box, 2x2x2 domains, rc 1.0 nm, "
                             "random local order"),
        Workload("water1M_4x4x4", 1_000_000, (21.5, 21.5, 21.5), (4, 4, 4), 1.2,
                 description="1,000,000 atoms, 21.5 nm box, 4x4x4 domains, rc 1.2 nm"),
        Workload("water3M_8x8x8", 3_000_000, (31.0, 31.0, 31.0), (8, 8, 8), 1.2,
                 rebuild_every=100,
                 description="3,000,000 atoms, 31 nm box, 8x8x8 domains, rc 1.2 nm, "
                             "rebuild every 100 exchanges after N(0, 0.01 nm) displacement"),
    )
}


def box_f32(box) -> np.ndarray:
    return np.asarray(box, dtype=np.float32)


def assign_domains(xyz: np.ndarray, box, grid) -> np.ndarray:
    """Domain id of each atom: the cell its position falls in.

    i_d = min(n_d - 1, floor(x_d * n_d / L_d)) in double, and
    D = ix + nx * (iy + ny * iz).
    """
    L = box_f32(box).astype(np.float64)
    n = np.asarray(grid, dtype=np.int64)
    x = xyz.astype(np.float64)
    cell = np.floor(x * n / L).astype(np.int64)
    cell = np.clip(cell, 0, n - 1)
    return (cell[:, 0] + n[0] * (cell[:, 1] + n[1] * cell[:, 2])).astype(np.int32)


def _wrap_f32(x64: np.ndarray, L: np.ndarray) -> np.ndarray:
    """Cast positions in [0, L) (double) to fp32; a value that rounds to L maps to 0."""
    x = x64.astype(np.float32)
    for d in range(3):
        col = x[:, d]
        col[col >= L[d]] = np.float32(0.0)
        col[col < 0] = np.float32(0.0)
    return x


def positions(n_atoms: int, box, seed: int) -> np.ndarray:
    """Uniform-random fp32 positions in [0, L) per component."""
    rng = np.random.default_rng(seed)
    L = box_f32(box)
    x64 = rng.random((n_atoms, 3)) * L.astype(np.float64)
    return _wrap_f32(x64, L)


def system(w: Workload | str, seed: int | None = None):
    """(xyz [N,3] f32, domain ids [N] i32) for a workload."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    s = w.seed if seed is None else seed
    xyz = positions(w.n_atoms, w.box, s)
    return xyz, assign_domains(xyz, w.box, w.grid)


def custom_system(n_atoms: int, box, grid, seed: int = 0):
    xyz = positions(n_atoms, box, seed)
    return xyz, assign_domains(xyz, box, grid)


def forces(n_slots: int, seed: int = 1) -> np.ndarray:
    """fp32 N(0, 1) force per component for every local slot."""
    rng = np.random.default_rng(seed)
    return rng.standard_normal((n_slots, 3)).astype(np.float32)


def integer_forces(n_slots: int, seed: int = 2, amp: int = 8) -> np.ndarray:
    """Small integer-valued fp32 forces in [-amp, amp] (sums stay exact in fp32)."""
    rng = np.random.default_rng(seed)
    return rng.integers(-amp, amp + 1, size=(n_slots, 3)).astype(np.float32)


def displaced(xyz: np.ndarray, box, grid, k: int, sigma: float = 0.01):
    """Positions after the k-th N(0, sigma) displacement (seed 1000 + k), wrapped
    into the box, and their recomputed domain ids."""
    rng = np.random.default_rng(1000 + k)
    L = box_f32(box)
    x64 = xyz.astype(np.float64) + rng.normal(0.0, sigma, size=xyz.shape)
    x64 = np.mod(x64, L.astype(np.float64))
    x = _wrap_f32(x64, L)
    return x, assign_domains(x, box, grid)
