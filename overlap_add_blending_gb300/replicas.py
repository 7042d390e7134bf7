"""Aggregation across replica ranks.

The tiled path has no data-path collective on one GPU: under torchrun each
rank runs its own replica of the workload and only the timing is combined.
The job's step time is the slowest rank's; its throughput counts the work
of every rank.
"""
from __future__ import annotations

from typing import Sequence, Tuple

import torch
import torch.distributed as dist


def combine(step_ms: Sequence[float], units_per_step: float, device=None) -> Tuple[list, float]:
    """Max over ranks of each timing in `step_ms`, and the units all ranks
    processed per step.  Without an initialised process group this is the
    identity (one replica)."""
    vals = [float(v) for v in step_ms]
    if not (dist.is_available() and dist.is_initialized()):
        return vals, float(units_per_step)
    world = dist.get_world_size()
    t = torch.tensor(vals + [float(units_per_step)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    mx = t[:-1].clone()
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    total = t[-1:].clone()
    dist.all_reduce(total, op=dist.ReduceOp.SUM)
    out = mx.cpu().tolist()
    assert len(out) == len(vals)
    return out, float(total.item()) if world > 0 else float(units_per_step)
