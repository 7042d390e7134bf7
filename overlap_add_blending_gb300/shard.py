"""The sharded blend across R ranks: tile exchange and per-rank slab blend.

"Tiled Data Parallelism (TDP)", What it is, gives tile t to rank t mod R and
sums the ranks' blended full-size buffers with one all_reduce.  Here each
rank instead owns a disjoint slab of output rows (tdp_shard_plan): it
receives, from their owners, the tiles that meet its slab but that it does
not own, and blends its slab alone (tdp_blend_slab).  The slabs, in rank
order along H, are the single-GPU blend bit for bit, and no full-size
buffer crosses the network.

The data plane is torch.distributed point-to-point (NCCL between GPUs, gloo
on CPU tensors): every tile is one contiguous block of the packed buffer,
sent whole by its owner to every rank whose slab it meets.
"""
from __future__ import annotations

from typing import List, Optional, Tuple

import torch
import torch.distributed as dist

from . import tdp


def exchange_plan(p: tdp.Plan, ranks: int) -> List[Tuple[int, int, int]]:
    """(tile, source rank, destination rank) of every transfer: each tile
    goes from its owner to each other rank whose slab it meets, in tile
    order, then destination order."""
    shards = [tdp.shard_plan(p, ranks, r) for r in range(ranks)]
    moves = []
    for t in range(p.T):
        src = t % ranks
        for dst in range(ranks):
            if dst != src and t in shards[dst].needed:
                moves.append((t, src, dst))
    return moves


def tile_block(p: tdp.Plan, tiles: torch.Tensor, B: int, C_: int, t: int) -> torch.Tensor:
    """Tile t's contiguous block of the packed buffer (a view)."""
    off = p.tile_offset(t, B, C_)
    (_, size) = p.box(t)
    n = B * C_ * size[0] * size[1] * size[2]
    return tiles[off:off + n]


def exchange_tiles(p: tdp.Plan, tiles: torch.Tensor, B: int, C_: int, group=None) -> int:
    """Fills, in this rank's packed buffer, every tile its slab needs from
    the tile's owner, and sends its own tiles to the ranks that need them.
    `tiles` holds valid data for this rank's owned tiles on entry.  Returns
    the bytes this rank received."""
    ranks = dist.get_world_size(group)
    rank = dist.get_rank(group)
    ops = []
    received = 0
    for t, src, dst in exchange_plan(p, ranks):
        blk = tile_block(p, tiles, B, C_, t)
        if src == rank:
            ops.append(dist.P2POp(dist.isend, blk, dist.get_global_rank(group, dst) if group else dst, group))
        elif dst == rank:
            ops.append(dist.P2POp(dist.irecv, blk, dist.get_global_rank(group, src) if group else src, group))
            received += blk.numel() * blk.element_size()
    if ops:
        for req in dist.batch_isend_irecv(ops):
            req.wait()
    return received


def sharded_blend(p: tdp.Plan, tiles: torch.Tensor, B: int, C_: int, group=None,
                  out: Optional[torch.Tensor] = None, out_dtype: Optional[torch.dtype] = None) -> torch.Tensor:
    """This rank's slab of the blend: the halo exchange, then tdp_blend_slab
    on the rank's rows.  Returns [B, C, F, row1 - row0, W]."""
    ranks = dist.get_world_size(group)
    rank = dist.get_rank(group)
    sh = tdp.shard_plan(p, ranks, rank)
    exchange_tiles(p, tiles, B, C_, group)
    return tdp.blend_slab(p, tiles, B, C_, sh.row0, sh.row1, out=out, out_dtype=out_dtype)
