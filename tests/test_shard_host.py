"""The sharded blend's host side: tdp_shard_plan against a reconstruction
from the plan's own intervals, the transfer list, and the halo exchange
between gloo ranks on CPU tensors.

Source: "Tiled Data Parallelism (TDP)", What it is (tile t goes to rank
t mod R; the ranks' blends are summed).  The slab form -- disjoint output
rows per rank, each rank receiving the tiles that meet its rows -- is this
library's reading of it."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from overlap_add_blending_gb300 import tdp
from overlap_add_blending_gb300.shard import exchange_plan, tile_block
from overlap_add_blending_gb300.workloads import WORKLOADS

PLANS = [
    ((16, 68, 120), ((2, 2), (4, 8), (4, 12)), False),     # the 4K tiling
    ((5, 37, 53), ((2, 1), (3, 5), (4, 6)), False),        # ragged
    ((1, 1, 21), ((1, 0), (1, 0), (4, 8)), True),          # H = 1
    ((3, 30, 10), ((1, 0), (5, 2), (1, 0)), False),       # many row tiles
]


def rows_of(p, t):
    (start, size) = p.box(t)
    return start[1], start[1] + size[1]


@pytest.mark.parametrize("dims,tiling,compat", PLANS)
@pytest.mark.parametrize("R", [1, 2, 3, 4, 7, 80])
def test_shard_plan_partitions_rows_and_lists_tiles(dims, tiling, compat, R):
    p = tdp.plan(dims, tiling, compat)
    H = dims[1]
    edges = []
    for r in range(R):
        sh = tdp.shard_plan(p, R, r)
        edges.append((sh.row0, sh.row1))
        assert sh.owned == tuple(t for t in range(p.T) if t % R == r)
        want = tuple(t for t in range(p.T) if sh.row0 < sh.row1 and rows_of(p, t)[0] < sh.row1
                     and rows_of(p, t)[1] > sh.row0)
        assert sh.needed == want
    # the slabs cover [0, H) once, in rank order, and differ in size by at most one row
    assert edges[0][0] == 0 and edges[-1][1] == H
    for (a0, a1), (b0, b1) in zip(edges, edges[1:]):
        assert a1 == b0 and a0 <= a1
    sizes = [b - a for a, b in edges]
    assert max(sizes) - min(sizes) <= 1


@pytest.mark.parametrize("dims,tiling,compat", PLANS)
def test_every_needed_tile_reaches_its_rank_once(dims, tiling, compat):
    p = tdp.plan(dims, tiling, compat)
    for R in (2, 3, 5):
        moves = exchange_plan(p, R)
        assert len(set(moves)) == len(moves)
        for r in range(R):
            sh = tdp.shard_plan(p, R, r)
            got = sorted(t for t, src, dst in moves if dst == r)
            assert got == sorted(set(sh.needed) - set(sh.owned))
            assert all(src == t % R and src != dst for t, src, dst in moves)


def test_shard_plan_rejects_bad_ranks():
    p = tdp.plan((4, 16, 16), ((1, 0), (2, 4), (2, 4)))
    for ranks, rank in ((0, 0), (2, 2), (2, -1)):
        with pytest.raises(tdp.TdpError):
            tdp.shard_plan(p, ranks, rank)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _exchange_worker(rank, world, port, case, q):
    import torch.distributed as dist
    from overlap_add_blending_gb300.shard import exchange_tiles
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dims, tiling, compat, B, C = case
        p = tdp.plan(dims, tiling, compat)
        n = p.tiles_numel(B, C)
        ref = torch.from_numpy(np.random.default_rng(11).standard_normal(n).astype(np.float32))
        local = torch.zeros(n, dtype=torch.float32)
        sh = tdp.shard_plan(p, world, rank)
        for t in sh.owned:
            tile_block(p, local, B, C, t).copy_(tile_block(p, ref, B, C, t))
        got = exchange_tiles(p, local, B, C)
        ok = True
        want_bytes = 0
        for t in range(p.T):
            blk, rb = tile_block(p, local, B, C, t), tile_block(p, ref, B, C, t)
            if t in sh.owned or t in sh.needed:
                ok &= bool(torch.equal(blk, rb))
            else:
                ok &= bool(torch.all(blk == 0))
            if t in sh.needed and t not in sh.owned:
                want_bytes += rb.numel() * 4
        q.put((rank, ok, got == want_bytes))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_halo_exchange_between_gloo_ranks(world):
    case = ((5, 37, 53), ((2, 1), (3, 5), (4, 6)), False, 2, 3)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_exchange_worker, args=(r, world, port, case, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    out = [q.get(timeout=180) for _ in range(world)]
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    for rank, ok, bytes_ok in out:
        assert ok, f"rank {rank}: a needed tile differs from its owner's, or an unneeded tile was written"
        assert bytes_ok, f"rank {rank}: received bytes differ from its halo"
