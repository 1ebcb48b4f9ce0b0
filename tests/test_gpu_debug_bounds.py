"""The MOE_DEBUG_BOUNDS build (libmoe_debug_bounds.so): the routing and
combine kernels check every expert and row index they use against its range
and record MOE_DEVICE_INDEX_OUT_OF_RANGE instead of making a bad access.

On valid inputs the checks must stay silent and the results must equal the
normal build's bit for bit; a bad expert index handed to the split-batch
finish is refused.  The debug build is loaded in a child process
(MOE_LIBRARY), since one process loads one build of the library."""
import json
import os
import subprocess
import sys

import pytest
import torch

from conftest import ROOT

pytestmark = pytest.mark.gpu

DEBUG_LIB = os.path.join(ROOT, "mixture_experts_layer_capacity_b300", "libmoe_debug_bounds.so")

CHILD = r'''
import json, sys
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
import numpy as np, torch
import parity
from mixture_experts_layer_capacity_b300 import binding as B
from mixture_experts_layer_capacity_b300.workloads import Workload
assert B.LIB_PATH.endswith("libmoe_debug_bounds.so"), B.LIB_PATH
cases = [
    ("multi_tile_top2", 1000, 256, 8, 384, 2, 192, 0, 0.0, "none"),
    ("t129_capacity", 129, 128, 8, 128, 2, 64, 1, 0.5, "normal_var2"),
    ("empty_experts_e64", 300, 128, 64, 128, 8, 0, 2, 0.0, "zipf1.1"),
    ("pair_tails_e128", 8200, 128, 128, 192, 8, 0, 2, 0.0, "zipf1.1"),
    ("fp32_top1", 256, 64, 4, 128, 1, 32, 2, 1.0, "none"),
    # E4M3 weights and activations: the dispatch gathers 1-byte codes
    ("a8_swap_capacity", 200, 192, 16, 320, 4, 0, 1, 0.75, "normal_var2"),
    ("a8_tiles_shared", 1000, 256, 8, 384, 2, 192, 0, 0.0, "none"),
]
out = {}
for name, T, D, E, F, k, S, mode, gamma, bias in cases:
    a8 = name.startswith("a8")
    w = Workload(name, T=T, D=D, E=E, F=F, k=k, S=S, mode=mode, gamma=gamma,
                 dtype="fp32" if name.startswith("fp32") else "bf16", alpha=0.01, bias=bias,
                 weights="e4m3" if a8 else "bf16", acts="e4m3" if a8 else "bf16")
    _, inp, outs, code = parity.run(w, seed=31)
    rep = parity.check(w, inp, outs, coverage=T > 4096, y_sample_n=96 if T > 4096 else None,
                       e4m3=a8, a8=a8)
    out[name] = dict(code=code, y_rel=rep["y_rel"],
                     y_sum=float(outs["y"].double().sum()))
print("RESULT " + json.dumps(out))
'''


def test_debug_bounds_build_is_silent_on_valid_layers():
    assert os.path.exists(DEBUG_LIB), "build with __graft_entry__.build()"
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, MOE_LIBRARY=DEBUG_LIB)
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], capture_output=True, text=True,
                       timeout=900, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("RESULT ")][-1]
    res = json.loads(line[len("RESULT "):])
    for name, v in res.items():
        assert v["code"] == 0, (name, v)
    print(res)
