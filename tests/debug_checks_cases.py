"""Runs the hot calls on the debug build (TDP_DEBUG_CHECKS=1 must be set
before the binding loads) and prints one JSON line: per case, whether the
outputs are right and the device error word after it.  Used by
test_gpu_debug_checks.py in a child process."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from oracle import tdp_oracle as O  # noqa: E402
from overlap_add_blending_gb300 import inputs, tdp  # noqa: E402
from overlap_add_blending_gb300.workloads import WORKLOADS  # noqa: E402

CASES = {
    "tiny": (WORKLOADS["tiny"].dims, WORKLOADS["tiny"].tiling, False, 1, 8, torch.float32),
    "ragged": ((5, 37, 53), ((2, 1), (3, 5), (4, 6)), False, 2, 3, torch.float32),
    "row_band": ((2, 300, 200), ((1, 0), (3, 20), (2, 16)), False, 1, 4, torch.bfloat16),
    "4k": (WORKLOADS["4k"].dims, WORKLOADS["4k"].tiling, False, 1, 16, torch.bfloat16),
    "triple": ((1, 21, 21), ((1, 0), (4, 8), (3, 8)), True, 1, 4, torch.float32),
}


def run(name):
    dims, tiling, compat, B, C, dt = CASES[name]
    dev = torch.device("cuda", 0)
    p = tdp.plan(dims, tiling, compat)
    rp = O.make_plan(dims, tiling, compat=compat)
    Xn = inputs.latent((B, C) + tuple(dims), seed=3)
    X = torch.from_numpy(Xn).to(dt).to(dev)
    tdp.device_error(clear=True)
    tiles = tdp.extract(p, X)
    out = tdp.blend(p, tiles, B, C)
    tok = tdp.extract_tokens(p, X) if (C * X.element_size()) % 16 == 0 else None
    slabs = [tdp.blend_slab(p, tiles, B, C, *(lambda s: (s.row0, s.row1))(tdp.shard_plan(p, 3, r)))
             for r in range(3)]
    torch.cuda.synchronize()
    ok = True
    ref = O.pack(O.extract(rp, X.float().cpu().double().numpy()))
    ok &= bool(np.array_equal(tiles.float().cpu().numpy().astype(np.float64), ref))
    ok &= bool(torch.equal(torch.cat(slabs, dim=3), out))
    if dt == torch.bfloat16 and not compat:
        ok &= bool(torch.equal(out, X))
    else:
        ok &= bool(torch.allclose(out.float(), X.float(), rtol=1e-5, atol=1e-5)) or compat
    if tok is not None:
        ok &= bool(np.array_equal(tok.float().cpu().numpy().astype(np.float64),
                                  O.pack(O.extract_tokens(rp, X.float().cpu().double().numpy()))))
    return {"ok": ok, "error_word": tdp.device_error(clear=True)}


if __name__ == "__main__":
    assert os.environ.get("TDP_DEBUG_CHECKS") == "1" and tdp.library_path().endswith("libtdp_debug.so")
    print(json.dumps({name: run(name) for name in CASES}))
