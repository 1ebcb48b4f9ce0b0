"""The MOE_TIMELINE build (libmoe_timeline.so): CTA 0 of each routed CTA-pair
GEMM launch stamps its units' MMA and epilogue phases, and every dispatch
block its phases.

The stamps must not change a result (the layer's y equals the normal
build's bit for bit), every recorded unit's and block's stamps must be in
the order the kernels run them (no dispatch block past the grid barrier
before every block has gated its tokens), and the pair's scheduler must
hand out all its full tiles before its swap units.  The timeline build is loaded in a child
process (MOE_LIBRARY), since one process loads one build of the library."""
import hashlib
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from conftest import ROOT
from mixture_experts_layer_capacity_b300 import binding as B
from mixture_experts_layer_capacity_b300 import timeline as TL
from mixture_experts_layer_capacity_b300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu

TL_LIB = os.path.join(ROOT, "mixture_experts_layer_capacity_b300", "libmoe_timeline.so")

# (name, T, D, E, F, k, S, mode, gamma, bias, E4M3 weights and activations)
CASES = [
    # 128 skewed experts: pair tiles, then many swap units; router GEMM
    # apart from the dispatch kernel
    ("pair_tails_e128_zipf", 8200, 128, 128, 192, 8, 0, 2, 0.0, "zipf1.1", False),
    # E4M3 pair tiles with drops and a shared expert (not recorded: dense);
    # the router fused into the dispatch kernel (E = 4)
    ("a8_pair_ragged_drops", 8200, 192, 4, 320, 2, 256, 1, 0.6, "normal_var2", True),
]


def _workload(case):
    name, T, D, E, F, k, S, mode, gamma, bias, a8 = case
    return Workload(name, T=T, D=D, E=E, F=F, k=k, S=S, mode=mode, gamma=gamma, dtype="bf16",
                    alpha=0.01, bias=bias, weights="e4m3" if a8 else "bf16",
                    acts="e4m3" if a8 else "bf16")


CHILD = r'''
import json, sys
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
from mixture_experts_layer_capacity_b300 import binding as B
from mixture_experts_layer_capacity_b300 import timeline as TL
import test_gpu_timeline as T
assert B.LIB_PATH.endswith("libmoe_timeline.so"), B.LIB_PATH
out = {}
for case in T.CASES:
    recs, outs = TL.collect(T._workload(case), seed=37)
    out[case[0]] = dict(
        y=T.y_digest(outs["y"]),
        status=B.read_device_status(B.config_of(T._workload(case)), outs["workspace"]),
        recs={r: v.tolist() for r, v in recs.items()})
print("RESULT " + json.dumps(out))
'''


def y_digest(y: torch.Tensor) -> str:
    return hashlib.sha256(y.detach().cpu().contiguous().view(torch.uint8).numpy().tobytes()).hexdigest()


def _normal_build_y(w, seed):
    cfg = B.config_of(w)
    inp = make_inputs(w, seed, "cuda")
    a8 = w.acts == "e4m3"
    if w.weights == "e4m3":
        inp = B.quantize_expert_weights(inp, a8=a8)
    outs = B.forward(cfg, inp)
    torch.cuda.synchronize()
    return y_digest(outs["y"])


def test_timeline_build_records_units_in_pipeline_order():
    assert os.path.exists(TL_LIB), "build with __graft_entry__.build()"
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, MOE_LIBRARY=TL_LIB)
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], capture_output=True, text=True,
                       timeout=900, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("RESULT ")][-1]
    res = json.loads(line[len("RESULT "):])
    for case in CASES:
        name = case[0]
        v = res[name]
        assert v["status"] == B.MOE_DEVICE_OK, name
        w = _workload(case)
        assert B.launch_plan(B.config_of(w))["pair_routed"], name
        # the stamps change no result
        assert v["y"] == _normal_build_y(w, 37), name
        for region in TL.REGIONS:
            rec = np.asarray(v["recs"][region], dtype=np.int64)
            assert len(rec) > 0, (name, region)
            assert set(rec[:, TL.IS_SWAP].tolist()) <= {0, 1}
            # MMA side: start <= has accumulator <= first stage full <= last issue
            for a, b in ((TL.MMA_START, TL.MMA_HAS_ACC), (TL.MMA_HAS_ACC, TL.FIRST_STAGE_FULL),
                         (TL.FIRST_STAGE_FULL, TL.LAST_MMA_ISSUED),
                         # epilogue side, and the accumulator is full only
                         # after the unit's last MMA was issued (same SM)
                         (TL.EPI_START, TL.EPI_ACC_FULL), (TL.EPI_ACC_FULL, TL.EPI_DONE),
                         (TL.LAST_MMA_ISSUED, TL.EPI_ACC_FULL)):
                assert (rec[:, a] <= rec[:, b]).all(), (name, region, a, b)
            # units follow one another on the pair: each starts no earlier
            # than the one before
            assert (np.diff(rec[:, TL.MMA_START]) >= 0).all()
            assert (np.diff(rec[:, TL.EPI_DONE]) >= 0).all()
            s = TL.summarize(rec)
            assert s["tiles_before_swaps"], (name, region)
            print(name, region, s["units"], s["swap_units"], s["bound"],
                  round(s["mma_issue_frac"], 3), round(s["epilogue_drain_frac"], 3))
        d = np.asarray(v["recs"]["dispatch"], dtype=np.int64)
        assert len(d) > 0, name
        # per block: start <= staged <= router <= gated <= ... <= copies done
        assert (np.diff(d, axis=1) >= 0).all(), name
        # the grid barrier: no block passes it before every block has
        # finished gating (1 us of slack for the timer's reads on other SMs)
        assert d[:, 5].min() >= d[:, 4].max() - 1000, name
        sd = TL.summarize_dispatch(d)
        print(name, "dispatch", sd["blocks"], round(sd["span_ns"] / 1e3, 1))
    # the skewed 128-expert layer has experts under 256 rows: swap units
    assert any(np.asarray(res["pair_tails_e128_zipf"]["recs"][r])[:, TL.IS_SWAP].any()
               for r in TL.REGIONS)
