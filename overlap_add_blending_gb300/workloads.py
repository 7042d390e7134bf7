"""Named workloads: latent shapes and per-axis (num_tiles, overlap) counts.

Pure data.  The shapes stand in for the LTX-2 stage-2 workloads by size
(there is no public dataset on this path); see the inputs module for how
values are drawn.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Tuple


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str                                   # "f32" or "bf16"
    B: int
    C: int
    dims: Tuple[int, int, int]                   # (F, H, W)
    tiling: Tuple[Tuple[int, int], ...]          # ((n_f, o_f), (n_h, o_h), (n_w, o_w))
    num_cond: int = 0                            # conditioning tokens
    num_cond_negative: int = 0                   # of which with a negative time start
    compat: bool = False


WORKLOADS = {
    "tiny": Workload("tiny", "f32", 1, 8, (4, 16, 16), ((1, 0), (2, 4), (2, 4)), 32, 8),
    "stage1": Workload("stage1", "bf16", 1, 128, (16, 16, 24), ((1, 0), (2, 4), (2, 6)), 64, 16),
    "fullres": Workload("fullres", "bf16", 1, 128, (16, 32, 48), ((1, 0), (2, 8), (2, 12)), 256, 64),
    "4k": Workload("4k", "bf16", 1, 128, (16, 68, 120), ((2, 2), (4, 8), (4, 12)), 256, 64),
    "strips": Workload("strips", "f32", 1, 16, (1, 128, 128), ((1, 0), (4, 8), (1, 0)), 0, 0),
    "grid": Workload("grid", "f32", 1, 16, (1, 128, 128), ((1, 0), (3, 8), (5, 8)), 0, 0),
}

# Guard-violating 1-D splits whose window-sum excess the mold issue measures.
SPLITS_1D = ((21, 2, 8), (21, 3, 8), (21, 4, 8))
