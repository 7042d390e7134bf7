"""Python binding of libtdp.so (C ABI in include/tdp.h).

Argument marshalling only: every step of the path runs in the library's
CUDA kernels (or, for planning and statistics, its host C++).  Tensors are
torch CUDA tensors; torch is used for device memory and streams.  Importing
this module raises ImportError when libtdp.so has not been built, and the
GPU entry points raise when given CPU tensors: there is no fallback path.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass
from typing import Optional, Sequence, Tuple

import torch

# TDP_DEBUG_CHECKS=1: the build with device index checks (build.py --debug)
_DEBUG = os.environ.get("TDP_DEBUG_CHECKS") == "1"
_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtdp_debug.so" if _DEBUG else "libtdp.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(f"{_LIB_PATH} is missing: build it with `python -m overlap_add_blending_gb300.build"
                      f"{' --debug' if _DEBUG else ''}`")
_lib = C.CDLL(_LIB_PATH)

MAX_PER_AXIS = 64
PLAN_UPSTREAM_COMPAT = 1
F32, BF16 = 0, 1

STATUS = {0: "ok", 1: "invalid argument", 2: "guard violated", 3: "too many tiles", 4: "alignment",
          5: "cuda error", 6: "unsupported"}


class TdpError(RuntimeError):
    def __init__(self, status: int, what: str):
        msg = _lib.tdp_status_str(status).decode()
        if status == 5:
            msg += f" (cudaError {_lib.tdp_last_cuda_error()})"
        super().__init__(f"{what}: {msg}")
        self.status = status


class DimCfg(C.Structure):
    _fields_ = [("num_tiles", C.c_int32), ("overlap", C.c_int32)]


class TileCountCfg(C.Structure):
    _fields_ = [("frames", DimCfg), ("height", DimCfg), ("width", DimCfg)]


class Plan(C.Structure):
    _fields_ = [
        ("dims", C.c_int32 * 3),
        ("num_tiles", C.c_int32 * 3),
        ("overlap", C.c_int32 * 3),
        ("stride", C.c_int32 * 3),
        ("start", (C.c_int32 * MAX_PER_AXIS) * 3),
        ("end", (C.c_int32 * MAX_PER_AXIS) * 3),
        ("prefix", (C.c_int32 * (MAX_PER_AXIS + 1)) * 3),
        ("max_cover", C.c_int32 * 3),
        ("total_tiles", C.c_int32),
        ("flags", C.c_uint32),
    ]

    # convenience views ------------------------------------------------
    @property
    def T(self) -> int:
        return int(self.total_tiles)

    def intervals(self, d: int):
        return [(int(self.start[d][i]), int(self.end[d][i])) for i in range(self.num_tiles[d])]

    def box(self, t: int) -> Tuple[Tuple[int, int, int], Tuple[int, int, int]]:
        start = (C.c_int32 * 3)()
        size = (C.c_int32 * 3)()
        _check(_lib.tdp_tile_box(C.byref(self), t, start, size), "tdp_tile_box")
        return tuple(start), tuple(size)

    def tile_offset(self, t: int, B: int, C_: int) -> int:
        return int(_lib.tdp_tile_offset(C.byref(self), t, B, C_))

    def tiles_numel(self, B: int, C_: int) -> int:
        return int(_lib.tdp_tiles_numel(C.byref(self), B, C_))

    def tokens_numel(self) -> int:
        """Total generated tokens over all tiles (sum of f_t * h_t * w_t)."""
        return int(_lib.tdp_tiles_numel(C.byref(self), 1, 1))


class LayoutCandidate(C.Structure):
    _fields_ = [
        ("num_tiles", C.c_int32 * 3),
        ("overlap", C.c_int32 * 3),
        ("window_volume", C.c_int64),
        ("decoded_volume", C.c_int64),
        ("heaviest_rank_volume", C.c_int64),
        ("seams", C.c_int32),
        ("role", C.c_int32),
    ]


ROLES = {0: "dominated", 1: "frontier", 2: "coarse", 3: "fine", 4: "balanced"}
SEARCH_NO_LIMITS = 2

_P = C.POINTER
_lib.tdp_plan.argtypes = [_P(C.c_int32 * 3), _P(TileCountCfg), C.c_uint32, _P(Plan)]
_lib.tdp_plan.restype = C.c_int
_lib.tdp_tile_offset.argtypes = [_P(Plan), C.c_int32, C.c_int32, C.c_int32]
_lib.tdp_tile_offset.restype = C.c_int64
_lib.tdp_tiles_numel.argtypes = [_P(Plan), C.c_int32, C.c_int32]
_lib.tdp_tiles_numel.restype = C.c_int64
_lib.tdp_tile_box.argtypes = [_P(Plan), C.c_int32, C.c_int32 * 3, C.c_int32 * 3]
_lib.tdp_tile_box.restype = C.c_int
_lib.tdp_plan_stats.argtypes = [_P(Plan), C.c_int32, _P(C.c_double), _P(C.c_int32), _P(C.c_double),
                                _P(C.c_double), _P(C.c_double)]
_lib.tdp_plan_stats.restype = C.c_int
_lib.tdp_extract.argtypes = [_P(Plan), C.c_int32, C.c_int32, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p]
_lib.tdp_extract.restype = C.c_int
_lib.tdp_blend.argtypes = [_P(Plan), C.c_int32, C.c_int32, C.c_int, C.c_void_p, C.c_int, C.c_void_p, C.c_void_p]
_lib.tdp_blend.restype = C.c_int
_lib.tdp_shard_plan.argtypes = [_P(Plan), C.c_int32, C.c_int32, _P(C.c_int32), _P(C.c_int32), C.c_void_p,
                                C.c_void_p]
_lib.tdp_shard_plan.restype = C.c_int
_lib.tdp_blend_slab.argtypes = [_P(Plan), C.c_int32, C.c_int32, C.c_int, C.c_void_p, C.c_int32, C.c_int32, C.c_int,
                                C.c_void_p, C.c_void_p]
_lib.tdp_blend_slab.restype = C.c_int
_lib.tdp_extract_tokens.argtypes = [_P(Plan), C.c_int32, C.c_int32, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p]
_lib.tdp_extract_tokens.restype = C.c_int
_lib.tdp_blend_tokens.argtypes = [_P(Plan), C.c_int32, C.c_int32, C.c_int, C.c_void_p, C.c_int, C.c_void_p,
                                  C.c_void_p]
_lib.tdp_blend_tokens.restype = C.c_int
_lib.tdp_window_sum.argtypes = [_P(Plan), C.c_void_p, C.c_void_p, C.c_void_p]
_lib.tdp_window_sum.restype = C.c_int
_lib.tdp_positions.argtypes = [_P(Plan), C.c_int32, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p]
_lib.tdp_positions.restype = C.c_int
_lib.tdp_cond_select.argtypes = [_P(Plan), C.c_int32, C.c_void_p, C.c_int32, C.c_void_p, C.c_int32,
                                 C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                 C.c_void_p, C.c_void_p]
_lib.tdp_cond_select.restype = C.c_int
_lib.tdp_tokens.argtypes = [_P(Plan), C.c_int32, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_int32,
                            C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                            C.c_void_p, C.c_void_p, C.c_void_p]
_lib.tdp_tokens.restype = C.c_int
_lib.tdp_extract_and_tokens.argtypes = [_P(Plan), C.c_int32, C.c_int32, C.c_int, C.c_void_p, C.c_void_p,
                                        C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p,
                                        C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                        C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int64, C.c_void_p]
_lib.tdp_extract_and_tokens.restype = C.c_int
_lib.tdp_extract_and_tokens_no_alloc.argtypes = [_P(Plan), C.c_int32, C.c_int32, C.c_int, C.c_void_p, C.c_void_p,
                                                 C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_int32,
                                                 C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                                 C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                                 C.c_void_p]
_lib.tdp_extract_and_tokens_no_alloc.restype = C.c_int
_lib.tdp_extract_and_tokens_workspace.argtypes = [_P(Plan), C.c_int32]
_lib.tdp_extract_and_tokens_workspace.restype = C.c_int64
_lib.tdp_cond_combine.argtypes = [_P(Plan), C.c_int32, C.c_int32, C.c_int32, C.c_int, C.c_void_p, C.c_void_p,
                                  C.c_void_p, C.c_int, C.c_void_p, C.c_void_p]
_lib.tdp_cond_combine.restype = C.c_int
_lib.tdp_balanced_tile_split.argtypes = [C.c_int32, _P(C.c_int32), _P(C.c_int32)]
_lib.tdp_balanced_tile_split.restype = C.c_int
_lib.tdp_search_layouts.argtypes = [_P(C.c_int32 * 3), C.c_int32, _P(DimCfg), C.c_int32, C.c_int32, C.c_uint32,
                                    _P(LayoutCandidate), C.c_int32, _P(C.c_int32)]
_lib.tdp_search_layouts.restype = C.c_int
_lib.tdp_device_error.argtypes = [_P(C.c_uint32), C.c_int32]
_lib.tdp_device_error.restype = C.c_int
_lib.tdp_status_str.argtypes = [C.c_int]
_lib.tdp_status_str.restype = C.c_char_p
_lib.tdp_last_cuda_error.argtypes = []
_lib.tdp_last_cuda_error.restype = C.c_int32
_lib.tdp_plan_struct_size.argtypes = []
_lib.tdp_plan_struct_size.restype = C.c_size_t


class LaunchGeometry(C.Structure):
    _fields_ = [(n, C.c_int32) for n in (
        "streaming", "band_rows", "nbands", "units", "grid", "stages", "stage_bytes", "max_runs", "shared_bytes",
        "off_hdr", "off_data", "chunks_per_row", "column_terms", "rows_per_thread", "threads", "run_slot",
        "table_bytes")] + [(n, C.c_int32 * 4) for n in ("class_first", "row_groups", "row_step")]

    def as_dict(self) -> dict:
        return {n: (list(getattr(self, n)) if n in ("class_first", "row_groups", "row_step") else int(getattr(self, n)))
                for n, _ in self._fields_}


_lib.tdp_launch_geometry.argtypes = [_P(Plan), C.c_int32, C.c_int32, C.c_int32, C.c_int, C.c_int, C.c_int32,
                                     _P(LaunchGeometry), _P(C.c_int32), C.c_int32, C.c_void_p, C.c_int32,
                                     _P(C.c_int32), C.c_int32, C.c_int32]
_lib.tdp_launch_geometry.restype = C.c_int

if _lib.tdp_plan_struct_size() != C.sizeof(Plan):
    raise ImportError("tdp_plan_t layout mismatch between libtdp.so and the binding")

EXPORTS = ("tdp_plan", "tdp_tile_offset", "tdp_tiles_numel", "tdp_tile_box", "tdp_plan_stats",
           "tdp_balanced_tile_split", "tdp_search_layouts",
           "tdp_extract", "tdp_positions", "tdp_cond_select", "tdp_tokens", "tdp_cond_combine", "tdp_blend",
           "tdp_extract_and_tokens", "tdp_extract_and_tokens_workspace", "tdp_extract_and_tokens_no_alloc",
           "tdp_shard_plan", "tdp_blend_slab",
           "tdp_extract_tokens", "tdp_blend_tokens", "tdp_window_sum",
           "tdp_launch_geometry", "tdp_device_error", "tdp_status_str", "tdp_last_cuda_error",
           "tdp_plan_struct_size")


def _check(status: int, what: str) -> None:
    if status != 0:
        raise TdpError(status, what)


def library_path() -> str:
    return _LIB_PATH


# ----------------------------------------------------------------- host calls
def plan(dims: Sequence[int], tiling: Sequence[Tuple[int, int]], compat: bool = False) -> Plan:
    """tdp_plan: dims = (F, H, W), tiling = ((n_f, o_f), (n_h, o_h), (n_w, o_w))."""
    d = (C.c_int32 * 3)(*[int(v) for v in dims])
    cfg = TileCountCfg(DimCfg(*tiling[0]), DimCfg(*tiling[1]), DimCfg(*tiling[2]))
    out = Plan()
    _check(_lib.tdp_plan(C.byref(d), C.byref(cfg), PLAN_UPSTREAM_COMPAT if compat else 0, C.byref(out)),
           "tdp_plan")
    return out


@dataclass
class PlanStats:
    decoded_area: float
    seams: int
    tile_fraction: float
    imbalance: float
    max_window_sum: float


def plan_stats(p: Plan, ranks: int = 1) -> PlanStats:
    a, tf, im, mw = C.c_double(), C.c_double(), C.c_double(), C.c_double()
    s = C.c_int32()
    _check(_lib.tdp_plan_stats(C.byref(p), ranks, C.byref(a), C.byref(s), C.byref(tf), C.byref(im), C.byref(mw)),
           "tdp_plan_stats")
    return PlanStats(a.value, s.value, tf.value, im.value, mw.value)


def launch_geometry(p: Plan, B: int, C_: int, blend: bool, in_dtype: torch.dtype, out_dtype: torch.dtype,
                    sm_count: int, tables: bool = False, rows: Optional[Tuple[int, int]] = None):
    """tdp_launch_geometry: (geometry dict, per-CTA first units) of a tdp_extract
    (blend False) or tdp_blend call (tdp_blend_slab with rows=(row0, row1))
    on a GPU with `sm_count` SMs; with tables=True also (the launch's plan
    tables as bytes, their section offsets in 16-byte words).  Host only."""
    row0, row1 = rows if rows is not None else (0, int(p.dims[1]))
    g = LaunchGeometry()
    starts = (C.c_int32 * 1025)()
    buf = (C.c_uint8 * 65536)()
    offs = (C.c_int32 * 7)()
    _check(_lib.tdp_launch_geometry(C.byref(p), B, C_, 1 if blend else 0, _dtype_code(in_dtype),
                                    _dtype_code(out_dtype), sm_count, C.byref(g), starts, len(starts),
                                    buf if tables else None, len(buf) if tables else 0, offs, row0, row1),
           "tdp_launch_geometry")
    d = g.as_dict()
    st = [int(v) for v in starts[:d["grid"] + 1]] if d["streaming"] else []
    if not tables:
        return d, st
    names = ("band", "frame", "row", "fcon", "wcon", "runs", "chunk")
    return d, st, bytes(buf[:d["table_bytes"]]), dict(zip(names, [int(v) for v in offs]))


def balanced_tile_split(ranks: int) -> Tuple[int, int]:
    """tdp_balanced_tile_split: (height tiles, width tiles) for `ranks` ranks."""
    h, w = C.c_int32(), C.c_int32()
    _check(_lib.tdp_balanced_tile_split(int(ranks), C.byref(h), C.byref(w)), "tdp_balanced_tile_split")
    return h.value, w.value


def search_layouts(dims: Sequence[int], ranks: int, frames: Tuple[int, int] = (1, 0), overlap_h: int = 0,
                   overlap_w: int = 0, compat: bool = False, limits: bool = True) -> list:
    """tdp_search_layouts: every candidate grid as a dict (counts, overlaps,
    volumes, seams, role), ordered by (n_h, n_w)."""
    d = (C.c_int32 * 3)(*[int(v) for v in dims])
    fr = DimCfg(*frames)
    flags = (PLAN_UPSTREAM_COMPAT if compat else 0) | (0 if limits else SEARCH_NO_LIMITS)
    n = C.c_int32()
    _check(_lib.tdp_search_layouts(C.byref(d), int(ranks), C.byref(fr), int(overlap_h), int(overlap_w), flags,
                                   None, 0, C.byref(n)), "tdp_search_layouts")
    buf = (LayoutCandidate * max(1, n.value))()
    _check(_lib.tdp_search_layouts(C.byref(d), int(ranks), C.byref(fr), int(overlap_h), int(overlap_w), flags,
                                   buf, n.value, C.byref(n)), "tdp_search_layouts")
    return [{"counts": tuple(c.num_tiles), "overlaps": tuple(c.overlap), "window_volume": c.window_volume,
             "decoded_volume": c.decoded_volume, "heaviest_rank_volume": c.heaviest_rank_volume,
             "seams": c.seams, "role": ROLES[c.role]} for c in buf[:n.value]]


# ----------------------------------------------------------------- device calls
_DT = {torch.float32: F32, torch.bfloat16: BF16}


def _stream(stream: Optional[torch.cuda.Stream]) -> C.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _dev(x: torch.Tensor, name: str, dtype=None) -> int:
    if not isinstance(x, torch.Tensor) or not x.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and x.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {x.dtype}")
    return x.data_ptr()


def _dtype_code(t: torch.dtype) -> int:
    if t not in _DT:
        raise TypeError(f"unsupported dtype {t}")
    return _DT[t]


def extract(p: Plan, latent: torch.Tensor, tiles: Optional[torch.Tensor] = None,
            stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """tdp_extract: latent [B, C, F, H, W] -> packed tiles (1-D, same dtype)."""
    if latent.dim() != 5 or tuple(latent.shape[2:]) != tuple(p.dims):
        raise ValueError(f"latent must be [B, C, {tuple(p.dims)}], got {tuple(latent.shape)}")
    B, Cc = int(latent.shape[0]), int(latent.shape[1])
    n = p.tiles_numel(B, Cc)
    if tiles is None:
        tiles = torch.empty(n, dtype=latent.dtype, device=latent.device)
    if tiles.numel() != n or tiles.dtype != latent.dtype:
        raise ValueError("tiles buffer has the wrong size or dtype")
    _check(_lib.tdp_extract(C.byref(p), B, Cc, _dtype_code(latent.dtype), _dev(latent, "latent"),
                            _dev(tiles, "tiles"), _stream(stream)), "tdp_extract")
    return tiles


def blend(p: Plan, tiles: torch.Tensor, B: int, C_: int, out: Optional[torch.Tensor] = None,
          out_dtype: Optional[torch.dtype] = None, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """tdp_blend: packed tiles -> latent [B, C, F, H, W]."""
    if tiles.numel() != p.tiles_numel(B, C_):
        raise ValueError("tiles has the wrong number of elements for this plan and batch")
    if out is None:
        out = torch.empty((B, C_) + tuple(p.dims), dtype=out_dtype or tiles.dtype, device=tiles.device)
    if tuple(out.shape) != (B, C_) + tuple(p.dims):
        raise ValueError("out has the wrong shape")
    _check(_lib.tdp_blend(C.byref(p), B, C_, _dtype_code(tiles.dtype), _dev(tiles, "tiles"),
                          _dtype_code(out.dtype), _dev(out, "out"), _stream(stream)), "tdp_blend")
    return out


@dataclass
class Shard:
    row0: int
    row1: int
    owned: Tuple[int, ...]      # tiles this rank owns (t mod ranks == rank)
    needed: Tuple[int, ...]     # tiles whose rows meet the rank's slab


def shard_plan(p: Plan, ranks: int, rank: int) -> Shard:
    """tdp_shard_plan: rank `rank`'s output slab and its owned / needed tiles."""
    r0, r1 = C.c_int32(), C.c_int32()
    owned = (C.c_uint8 * max(1, p.T))()
    needed = (C.c_uint8 * max(1, p.T))()
    _check(_lib.tdp_shard_plan(C.byref(p), ranks, rank, C.byref(r0), C.byref(r1), owned, needed), "tdp_shard_plan")
    return Shard(r0.value, r1.value, tuple(t for t in range(p.T) if owned[t]),
                 tuple(t for t in range(p.T) if needed[t]))


def blend_slab(p: Plan, tiles: torch.Tensor, B: int, C_: int, row0: int, row1: int,
               out: Optional[torch.Tensor] = None, out_dtype: Optional[torch.dtype] = None,
               stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """tdp_blend_slab: packed tiles -> rows [row0, row1) of the blend, [B, C, F, row1-row0, W]."""
    if tiles.numel() != p.tiles_numel(B, C_):
        raise ValueError("tiles has the wrong number of elements for this plan and batch")
    shape = (B, C_, p.dims[0], row1 - row0, p.dims[2])
    if out is None:
        out = torch.empty(shape, dtype=out_dtype or tiles.dtype, device=tiles.device)
    if tuple(out.shape) != shape:
        raise ValueError("out has the wrong shape")
    _check(_lib.tdp_blend_slab(C.byref(p), B, C_, _dtype_code(tiles.dtype), _dev(tiles, "tiles"), row0, row1,
                               _dtype_code(out.dtype), _dev(out, "out"), _stream(stream)), "tdp_blend_slab")
    return out


def extract_tokens(p: Plan, latent: torch.Tensor, tokens: Optional[torch.Tensor] = None,
                   stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """tdp_extract_tokens: latent [B, C, F, H, W] -> packed token-major tiles
    (1-D, same dtype; tile t is [B, N_t, C] at tile_offset(t, B, C))."""
    if latent.dim() != 5 or tuple(latent.shape[2:]) != tuple(p.dims):
        raise ValueError(f"latent must be [B, C, {tuple(p.dims)}], got {tuple(latent.shape)}")
    B, Cc = int(latent.shape[0]), int(latent.shape[1])
    n = p.tiles_numel(B, Cc)
    if tokens is None:
        tokens = torch.empty(n, dtype=latent.dtype, device=latent.device)
    if tokens.numel() != n or tokens.dtype != latent.dtype:
        raise ValueError("tokens buffer has the wrong size or dtype")
    _check(_lib.tdp_extract_tokens(C.byref(p), B, Cc, _dtype_code(latent.dtype), _dev(latent, "latent"),
                                   _dev(tokens, "tokens"), _stream(stream)), "tdp_extract_tokens")
    return tokens


def blend_tokens(p: Plan, tokens: torch.Tensor, B: int, C_: int, out: Optional[torch.Tensor] = None,
                 out_dtype: Optional[torch.dtype] = None, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """tdp_blend_tokens: packed token-major tiles -> latent [B, C, F, H, W]."""
    if tokens.numel() != p.tiles_numel(B, C_):
        raise ValueError("tokens has the wrong number of elements for this plan and batch")
    if out is None:
        out = torch.empty((B, C_) + tuple(p.dims), dtype=out_dtype or tokens.dtype, device=tokens.device)
    if tuple(out.shape) != (B, C_) + tuple(p.dims):
        raise ValueError("out has the wrong shape")
    _check(_lib.tdp_blend_tokens(C.byref(p), B, C_, _dtype_code(tokens.dtype), _dev(tokens, "tokens"),
                                 _dtype_code(out.dtype), _dev(out, "out"), _stream(stream)), "tdp_blend_tokens")
    return out


def window_sum(p: Plan, max_dev: Optional[torch.Tensor] = None, sum_out: Optional[torch.Tensor] = None,
               want_sum: bool = False, device=None, stream: Optional[torch.cuda.Stream] = None):
    """tdp_window_sum: returns (max |S-1| as a 1-element tensor, S or None)."""
    device = device or torch.device("cuda")
    if max_dev is None:
        max_dev = torch.empty(4, dtype=torch.float32, device=device)
    if sum_out is None and want_sum:
        sum_out = torch.empty(tuple(p.dims), dtype=torch.float32, device=device)
    _check(_lib.tdp_window_sum(C.byref(p), _dev(max_dev, "max_dev", torch.float32),
                               None if sum_out is None else _dev(sum_out, "sum_out", torch.float32),
                               _stream(stream)), "tdp_window_sum")
    return max_dev[:1], sum_out


def positions(p: Plan, gen_pos: torch.Tensor, normalize: bool = True, tile_pos: Optional[torch.Tensor] = None,
              offsets: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None):
    """tdp_positions: gen_pos int32 [B, 3, N, 2] -> (packed tile positions, offsets [T, B, 3])."""
    B = int(gen_pos.shape[0])
    N = p.dims[0] * p.dims[1] * p.dims[2]
    if tuple(gen_pos.shape) != (B, 3, N, 2):
        raise ValueError("gen_pos must be [B, 3, F*H*W, 2]")
    if tile_pos is None:
        tile_pos = torch.empty(6 * B * p.tokens_numel(), dtype=torch.int32, device=gen_pos.device)
    if offsets is None:
        offsets = torch.empty((p.T, B, 3), dtype=torch.int32, device=gen_pos.device)
    _check(_lib.tdp_positions(C.byref(p), B, _dev(gen_pos, "gen_pos", torch.int32), 1 if normalize else 0,
                              _dev(tile_pos, "tile_pos", torch.int32), _dev(offsets, "offsets", torch.int32),
                              _stream(stream)), "tdp_positions")
    return tile_pos, offsets


def tile_positions_view(p: Plan, tile_pos: torch.Tensor, B: int, t: int) -> torch.Tensor:
    """[B, 3, N_t, 2] view of tile t inside the packed positions buffer."""
    (_, size) = p.box(t)
    n_t = size[0] * size[1] * size[2]
    off = 6 * B * (p.tile_offset(t, 1, 1))
    return tile_pos[off:off + 6 * B * n_t].view(B, 3, n_t, 2)


def cond_select(p: Plan, gen_pos: torch.Tensor, cond_pos: torch.Tensor, normalize: bool = True,
                with_lists: bool = True, out: Optional[dict] = None,
                stream: Optional[torch.cuda.Stream] = None) -> dict:
    """tdp_cond_select.  Returns a dict of device tensors: extent [T,B,3,2],
    keep [T,B,M] uint8, count [B,M], weight [B,M], and (with_lists) kept_idx
    [T,B,M], num_kept [T,B], tile_cond_pos [T,B,3,M,2]."""
    B, _, M, _ = cond_pos.shape
    dev = gen_pos.device
    T = p.T
    o = out if out is not None else {}
    if not o:
        o["extent"] = torch.empty((T, B, 3, 2), dtype=torch.int32, device=dev)
        o["keep"] = torch.empty((T, B, M), dtype=torch.uint8, device=dev)
        o["count"] = torch.empty((B, M), dtype=torch.int32, device=dev)
        o["weight"] = torch.empty((B, M), dtype=torch.float32, device=dev)
        if with_lists:
            o["kept_idx"] = torch.empty((T, B, M), dtype=torch.int32, device=dev)
            o["num_kept"] = torch.empty((T, B), dtype=torch.int32, device=dev)
            o["tile_cond_pos"] = torch.empty((T, B, 3, M, 2), dtype=torch.int32, device=dev)

    def opt(name, dtype):
        return _dev(o[name], name, dtype) if name in o else None

    _check(_lib.tdp_cond_select(C.byref(p), int(B), _dev(gen_pos, "gen_pos", torch.int32), int(M),
                                _dev(cond_pos, "cond_pos", torch.int32), 1 if normalize else 0,
                                _dev(o["extent"], "extent", torch.int32), _dev(o["keep"], "keep", torch.uint8),
                                _dev(o["count"], "count", torch.int32), _dev(o["weight"], "weight", torch.float32),
                                opt("kept_idx", torch.int32), opt("num_kept", torch.int32),
                                opt("tile_cond_pos", torch.int32), _stream(stream)), "tdp_cond_select")
    return o


def tokens(p: Plan, gen_pos: torch.Tensor, cond_pos: torch.Tensor, normalize: bool = True,
           with_lists: bool = True, out: Optional[dict] = None,
           stream: Optional[torch.cuda.Stream] = None) -> dict:
    """tdp_tokens: positions and conditioning selection in one launch.  Returns
    the cond_select dict plus "tile_pos" (packed) and "offsets" [T, B, 3]."""
    B = int(gen_pos.shape[0])
    M = int(cond_pos.shape[2])
    N = p.dims[0] * p.dims[1] * p.dims[2]
    if tuple(gen_pos.shape) != (B, 3, N, 2) or tuple(cond_pos.shape) != (B, 3, M, 2):
        raise ValueError("gen_pos must be [B, 3, F*H*W, 2] and cond_pos [B, 3, M, 2]")
    o = out if out is not None else {}
    if not o:
        o.update(token_outputs(p, B, M, gen_pos.device, with_lists))

    def opt(name, dtype):
        return _dev(o[name], name, dtype) if name in o else None

    _check(_lib.tdp_tokens(C.byref(p), B, _dev(gen_pos, "gen_pos", torch.int32), 1 if normalize else 0,
                           opt("tile_pos", torch.int32), opt("offsets", torch.int32), M,
                           _dev(cond_pos, "cond_pos", torch.int32) if M > 0 else None,
                           opt("extent", torch.int32), opt("keep", torch.uint8), opt("count", torch.int32),
                           opt("weight", torch.float32), opt("kept_idx", torch.int32), opt("num_kept", torch.int32),
                           opt("tile_cond_pos", torch.int32), opt("slot_of", torch.int32), _stream(stream)),
           "tdp_tokens")
    return o


def token_outputs(p: Plan, B: int, M: int, device, with_lists: bool = True) -> dict:
    """Empty device buffers for every output of tdp_tokens (the dict tokens
    and extract_and_tokens fill)."""
    T = p.T
    o = {"tile_pos": torch.empty(6 * B * p.tokens_numel(), dtype=torch.int32, device=device),
         "offsets": torch.empty((T, B, 3), dtype=torch.int32, device=device),
         "extent": torch.empty((T, B, 3, 2), dtype=torch.int32, device=device),
         "keep": torch.empty((T, B, M), dtype=torch.uint8, device=device),
         "count": torch.empty((B, M), dtype=torch.int32, device=device),
         "weight": torch.empty((B, M), dtype=torch.float32, device=device)}
    if with_lists:
        o["kept_idx"] = torch.empty((T, B, M), dtype=torch.int32, device=device)
        o["num_kept"] = torch.empty((T, B), dtype=torch.int32, device=device)
        o["tile_cond_pos"] = torch.empty((T, B, 3, M, 2), dtype=torch.int32, device=device)
        o["slot_of"] = torch.empty((T, B, M), dtype=torch.int32, device=device)
    return o


def extract_and_tokens_workspace(p: Plan, B: int) -> int:
    """tdp_extract_and_tokens_workspace: bytes of device workspace the call needs."""
    n = int(_lib.tdp_extract_and_tokens_workspace(C.byref(p), int(B)))
    if n < 0:
        raise ValueError("invalid plan or batch")
    return n


def extract_and_tokens(p: Plan, latent: torch.Tensor, gen_pos: torch.Tensor, cond_pos: torch.Tensor,
                       tiles: Optional[torch.Tensor] = None, tok: Optional[dict] = None,
                       max_dev: Optional[torch.Tensor] = None, window_max: bool = True,
                       workspace: Optional[torch.Tensor] = None, normalize: bool = True,
                       stream: Optional[torch.cuda.Stream] = None):
    """tdp_extract_and_tokens: the tiles, every output of tokens() and (unless
    window_max is False) max |S-1| in two launches.  `tok` as token_outputs()
    makes it (keys left out are not written; an empty or missing dict is
    filled with new buffers); max_dev a 4-float buffer; workspace a byte
    buffer of extract_and_tokens_workspace() bytes (made here when None).
    Returns (tiles, tok, max_dev[:1] or None)."""
    if latent.dim() != 5 or tuple(latent.shape[2:]) != tuple(p.dims):
        raise ValueError(f"latent must be [B, C, {tuple(p.dims)}], got {tuple(latent.shape)}")
    B, Cc = int(latent.shape[0]), int(latent.shape[1])
    M = int(cond_pos.shape[2])
    N = p.dims[0] * p.dims[1] * p.dims[2]
    if tuple(gen_pos.shape) != (B, 3, N, 2) or tuple(cond_pos.shape) != (B, 3, M, 2):
        raise ValueError("gen_pos must be [B, 3, F*H*W, 2] and cond_pos [B, 3, M, 2]")
    n = p.tiles_numel(B, Cc)
    if tiles is None:
        tiles = torch.empty(n, dtype=latent.dtype, device=latent.device)
    if tiles.numel() != n or tiles.dtype != latent.dtype:
        raise ValueError("tiles buffer has the wrong size or dtype")
    o = tok if tok is not None else {}
    if not o:
        o.update(token_outputs(p, B, M, latent.device))
    if window_max and max_dev is None:
        max_dev = torch.empty(4, dtype=torch.float32, device=latent.device)
    if workspace is None:
        workspace = torch.empty(max(16, extract_and_tokens_workspace(p, B)), dtype=torch.uint8, device=latent.device)

    def opt(name, dtype):
        return _dev(o[name], name, dtype) if name in o else None

    _check(_lib.tdp_extract_and_tokens(C.byref(p), B, Cc, _dtype_code(latent.dtype), _dev(latent, "latent"),
                                       _dev(tiles, "tiles"), _dev(gen_pos, "gen_pos", torch.int32),
                                       1 if normalize else 0, opt("tile_pos", torch.int32),
                                       opt("offsets", torch.int32), M,
                                       _dev(cond_pos, "cond_pos", torch.int32) if M > 0 else None,
                                       opt("extent", torch.int32), opt("keep", torch.uint8),
                                       opt("count", torch.int32), opt("weight", torch.float32),
                                       opt("kept_idx", torch.int32), opt("num_kept", torch.int32),
                                       opt("tile_cond_pos", torch.int32), opt("slot_of", torch.int32),
                                       _dev(max_dev, "max_dev", torch.float32) if window_max else None,
                                       _dev(workspace, "workspace", torch.uint8), workspace.numel(),
                                       _stream(stream)), "tdp_extract_and_tokens")
    return tiles, o, (max_dev[:1] if window_max else None)


def extract_and_tokens_no_alloc(p: Plan, latent: torch.Tensor, gen_pos: torch.Tensor, cond_pos: torch.Tensor,
                                tiles: torch.Tensor, tok: dict, max_dev: Optional[torch.Tensor] = None,
                                normalize: bool = True, stream: Optional[torch.cuda.Stream] = None):
    """tdp_extract_and_tokens_no_alloc: extract_and_tokens into the caller's
    buffers (tiles, tok as token_outputs() makes it, max_dev a 4-float buffer
    or None) with the library's own scratch; this binding allocates nothing
    either."""
    B, Cc = int(latent.shape[0]), int(latent.shape[1])
    M = int(cond_pos.shape[2])

    def opt(name, dtype):
        return _dev(tok[name], name, dtype) if name in tok else None

    _check(_lib.tdp_extract_and_tokens_no_alloc(
        C.byref(p), B, Cc, _dtype_code(latent.dtype), _dev(latent, "latent"), _dev(tiles, "tiles"),
        _dev(gen_pos, "gen_pos", torch.int32), 1 if normalize else 0, opt("tile_pos", torch.int32),
        opt("offsets", torch.int32), M, _dev(cond_pos, "cond_pos", torch.int32) if M > 0 else None,
        opt("extent", torch.int32), opt("keep", torch.uint8), opt("count", torch.int32),
        opt("weight", torch.float32), opt("kept_idx", torch.int32), opt("num_kept", torch.int32),
        opt("tile_cond_pos", torch.int32), opt("slot_of", torch.int32),
        None if max_dev is None else _dev(max_dev, "max_dev", torch.float32), _stream(stream)),
        "tdp_extract_and_tokens_no_alloc")


def cond_combine(p: Plan, tile_cond_out: torch.Tensor, slot_of: torch.Tensor, weight: torch.Tensor,
                 out: Optional[torch.Tensor] = None, out_dtype: Optional[torch.dtype] = None,
                 stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """tdp_cond_combine: tile_cond_out [T, B, M, D] (bf16/fp32, kept order),
    slot_of int32 [T, B, M], weight float [B, M] -> out [B, M, D]."""
    T, B, M, D = (int(v) for v in tile_cond_out.shape)
    if T != p.T or tuple(slot_of.shape) != (T, B, M) or tuple(weight.shape) != (B, M):
        raise ValueError("tile_cond_out [T,B,M,D], slot_of [T,B,M] and weight [B,M] must agree with the plan")
    odt = out_dtype or tile_cond_out.dtype
    if out is None:
        out = torch.empty((B, M, D), dtype=odt, device=tile_cond_out.device)
    _check(_lib.tdp_cond_combine(C.byref(p), B, M, D, _DT[tile_cond_out.dtype],
                                 _dev(tile_cond_out, "tile_cond_out", tile_cond_out.dtype),
                                 _dev(slot_of, "slot_of", torch.int32), _dev(weight, "weight", torch.float32),
                                 _DT[out.dtype], _dev(out, "out", out.dtype), _stream(stream)), "tdp_cond_combine")
    return out


def device_error(clear: bool = True) -> int:
    v = C.c_uint32()
    _check(_lib.tdp_device_error(C.byref(v), 1 if clear else 0), "tdp_device_error")
    return int(v.value)
