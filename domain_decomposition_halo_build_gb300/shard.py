"""Host side of the sharded data plane (include/halo.h, halo_shard ...).

The domains of a system are split into z-slabs, one per shard; a shard would
be one GPU's share of the system ("Redesigning GROMACS Halo Exchange ...",
section 3: domains on several GPUs, pulses between them).  These functions
hold the partition rule (the same as halo_shard's), the shard's slot range in
the dense local layout, and the exchange of every rank's layout and buffer
handles that ranks need before they can address each other's halo slices.
They run on the host only; nothing here touches a GPU.
"""
from __future__ import annotations

from typing import Dict, List, Sequence


def partition(grid: Sequence[int], n_shards: int) -> List[tuple]:
    """(first_domain, n_domains) of every shard: shard k takes the z layers
    [k*nz/n, (k+1)*nz/n); domain id = ix + nx*(iy + ny*iz), so each slab is
    a contiguous id range."""
    nx, ny, nz = (int(g) for g in grid)
    if not 1 <= n_shards <= min(8, nz):
        raise ValueError("n_shards must be in [1, min(8, n_z)]")
    layer = nx * ny
    cuts = [(k * nz // n_shards) * layer for k in range(n_shards + 1)]
    return [(cuts[k], cuts[k + 1] - cuts[k]) for k in range(n_shards)]


def shard_of_domain(grid: Sequence[int], n_shards: int, domain: int) -> int:
    for k, (first, count) in enumerate(partition(grid, n_shards)):
        if first <= domain < first + count:
            return k
    raise ValueError("domain out of range")


def slot_ranges(n_local: Sequence[int], parts: List[tuple]) -> List[tuple]:
    """(first_slot, n_slots) of every shard in the dense local layout (domains
    one after another, n_local[D] slots each)."""
    base = [0]
    for v in n_local:
        base.append(base[-1] + int(v))
    return [(base[first], base[first + count] - base[first]) for first, count in parts]


def exchange_layouts(layout: Dict, handle: bytes, group=None) -> List[Dict]:
    """Every rank's layout and buffer handle, in rank order (all ranks call
    it).  layout: this rank's {"shard", "first_domain", "n_domains",
    "first_slot", "n_local"}; handle: an opaque blob naming this rank's shard
    buffer and counters to its peers."""
    import torch.distributed as dist
    mine = dict(layout, handle=bytes(handle))
    out: List = [None] * dist.get_world_size(group)
    dist.all_gather_object(out, mine, group=group)
    return out


def owner_of_slot(table: List[Dict], slot: int) -> int:
    """Rank whose shard holds dense slot `slot` (table: exchange_layouts)."""
    for r, t in enumerate(table):
        if t["first_slot"] <= slot < t["first_slot"] + t["n_local"]:
            return r
    raise ValueError("slot outside every shard")
