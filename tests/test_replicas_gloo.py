"""The N > 1 bench path: replicas combine their timings over a process group
(max of step times, sum of work).  Two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist

    from overlap_add_blending_gb300.replicas import combine
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [1.0 + rank, 5.0 - rank, 0.25 * (rank + 1)]
        mx, units = combine(ms, units_per_step=100.0 + rank)
        q.put((rank, mx, units))
    finally:
        dist.destroy_process_group()


def test_combine_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, units in out:
        assert mx == [2.0, 5.0, 0.5]
        assert units == 201.0


def test_combine_single_process_is_identity():
    from overlap_add_blending_gb300.replicas import combine
    mx, units = combine([3.0, 4.0], 7.0)
    assert mx == [3.0, 4.0] and units == 7.0
