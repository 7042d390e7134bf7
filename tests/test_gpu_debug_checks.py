"""The debug build (TDP_DEBUG_CHECKS=1): every global and shared index of
the hot kernels' accesses is checked, and a failed check sets bit 8 of the
device error word instead of making the access.  On the tiny, ragged,
row-band, 4K and compat-triple cases the checks must all pass (the word
stays 0) and the outputs must still be right.  Runs the cases in a child
process that loads libtdp_debug.so."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_debug_build_index_checks_pass():
    from overlap_add_blending_gb300 import build
    build.build(debug=True)
    env = dict(os.environ, TDP_DEBUG_CHECKS="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_checks_cases.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    res = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1])
    for name, v in res.items():
        assert v["error_word"] == 0, f"{name}: device error word {v['error_word']:#x} on the debug build"
        assert v["ok"], f"{name}: wrong outputs on the debug build"
