"""Per-unit timeline of the routed CTA-pair expert GEMMs and per-block
timeline of the dispatch kernel.

    python -m mixture_experts_layer_capacity_b300.timeline --workload dsv3_prefill [--json]

Loads ``libmoe_timeline.so`` (the library built with ``-DMOE_TIMELINE``;
``python -m mixture_experts_layer_capacity_b300.build --timeline``), runs a
few forward passes of the named layer, and reads back the stamps that CTA 0
of the routed gate/up and down-projection pair launches wrote for each of its
units (a 256-row pair tile or a swap unit).  The summary says where one CTA
pair's time goes: the MMA thread waiting for a free accumulator or for its
first operand stage, issuing the unit's MMAs, and the epilogue warps waiting
for the accumulator and draining it to HBM.  A GEMM whose epilogue drain is
longer than its MMA issue span is bound by its epilogue, not by the tensor
pipe.  For the dispatch kernel it gives, per phase, the median and the
latest time (over the blocks) at which a block finished it, counted from
the first block's start.

The stamps are the GPU's global nanosecond timer; each record holds eight
words (see ``moe_timeline_read`` in include/moe.h).  The instrumented library
computes the same results as the normal one, bit for bit, but its stores add
a little time per unit, so its timings explain a profile rather than replace
the bench.
"""
from __future__ import annotations

import argparse
import json
import os
import sys

import numpy as np

WORDS_PER_UNIT = 8
MAX_UNITS = 4096
REGIONS = ("gemm1", "gemm2")   # gate/up, down projection

# word index of each stamp in a unit's record
MMA_START, MMA_HAS_ACC, FIRST_STAGE_FULL, LAST_MMA_ISSUED = 0, 1, 2, 3
EPI_ACC_FULL, EPI_DONE, IS_SWAP, EPI_START = 4, 5, 6, 7

# the dispatch kernel's per-block records follow the GEMM regions
DISPATCH_BASE = len(REGIONS) * MAX_UNITS * WORDS_PER_UNIT
# word index -> phase a dispatch block has finished at that stamp
DISPATCH_PHASES = {1: "rows_staged", 2: "router", 3: "gated_first_chunk", 4: "gating",
                   5: "grid_barrier", 6: "segment_tables", 7: "row_copies"}

# phase name -> (end word, start word)
PHASES = {
    "mma_waits_accumulator": (MMA_HAS_ACC, MMA_START),
    "mma_waits_first_stage": (FIRST_STAGE_FULL, MMA_HAS_ACC),
    "mma_issue": (LAST_MMA_ISSUED, FIRST_STAGE_FULL),
    "epilogue_waits_accumulator": (EPI_ACC_FULL, EPI_START),
    "epilogue_drain": (EPI_DONE, EPI_ACC_FULL),
}


def units(words: np.ndarray, region: int) -> np.ndarray:
    """The recorded units of one region as an (n, 8) int64 array, in the
    order CTA 0 ran them.  A unit counts once both its MMA side and its
    epilogue side have written their stamps; recording stops at the first
    unit that has not."""
    r = np.asarray(words, dtype=np.uint64)
    base = region * MAX_UNITS * WORDS_PER_UNIT
    rec = r[base:base + MAX_UNITS * WORDS_PER_UNIT].reshape(MAX_UNITS, WORDS_PER_UNIT)
    done = (rec[:, MMA_START] != 0) & (rec[:, EPI_DONE] != 0)
    n = int(np.argmin(done)) if not done.all() else MAX_UNITS
    return rec[:n].astype(np.int64)


def dispatch_blocks(words: np.ndarray) -> np.ndarray:
    """The dispatch kernel's per-block records as an (n, 8) int64 array,
    block order; recording stops at the first block that did not start."""
    r = np.asarray(words, dtype=np.uint64)
    rec = r[DISPATCH_BASE:DISPATCH_BASE + MAX_UNITS * WORDS_PER_UNIT]
    if len(rec) < MAX_UNITS * WORDS_PER_UNIT:
        return np.zeros((0, WORDS_PER_UNIT), dtype=np.int64)
    rec = rec.reshape(MAX_UNITS, WORDS_PER_UNIT)
    started = rec[:, 0] != 0
    n = int(np.argmin(started)) if not started.all() else MAX_UNITS
    return rec[:n].astype(np.int64)


def summarize_dispatch(rec: np.ndarray) -> dict:
    """Per phase, the median and the maximum over blocks of the time (ns)
    from the first block's start to the block's stamp, and the span to the
    last row copy."""
    rec = np.asarray(rec, dtype=np.int64)
    if len(rec) == 0:
        return {"blocks": 0}
    t0 = int(rec[:, 0].min())
    out = {"blocks": len(rec), "span_ns": int(rec[:, 7].max() - t0), "phases": {}}
    for word, name in DISPATCH_PHASES.items():
        d = rec[:, word] - t0
        out["phases"][name] = {"median_ns": float(np.median(d)), "max_ns": int(d.max())}
    return out


def summarize(rec: np.ndarray) -> dict:
    """Phase durations of one region's units (ns): mean and total over all
    units and the means over pair tiles and swap units apart, the span from
    the first unit's start to the last epilogue's end, and the fraction of
    that span the MMA issue and the epilogue drain each fill."""
    rec = np.asarray(rec, dtype=np.int64)
    n = len(rec)
    if n == 0:
        return {"units": 0}
    swap = rec[:, IS_SWAP] == 1
    span = int(rec[:, EPI_DONE].max() - rec[:, MMA_START].min())
    out = {"units": n, "swap_units": int(swap.sum()), "span_ns": span, "phases": {}}
    for name, (end, start) in PHASES.items():
        d = rec[:, end] - rec[:, start]
        out["phases"][name] = {
            "mean_ns": float(d.mean()),
            "total_ns": int(d.sum()),
            "tile_mean_ns": float(d[~swap].mean()) if (~swap).any() else None,
            "swap_mean_ns": float(d[swap].mean()) if swap.any() else None,
        }
    ph = out["phases"]
    out["mma_issue_frac"] = ph["mma_issue"]["total_ns"] / span if span else 0.0
    out["epilogue_drain_frac"] = ph["epilogue_drain"]["total_ns"] / span if span else 0.0
    out["bound"] = ("epilogue" if ph["epilogue_drain"]["mean_ns"] > ph["mma_issue"]["mean_ns"]
                    else "mma")
    # the scheduler hands a pair all its full tiles before its swap units
    out["tiles_before_swaps"] = bool(not swap.any() or not (~swap[int(np.argmax(swap)):]).any())
    return out


def format_summary(name: str, summ: dict) -> str:
    lines = [f"== {name}"]
    d = summ.get("dispatch", {"blocks": 0})
    if d["blocks"]:
        lines.append(f" dispatch: {d['blocks']} blocks, span {d['span_ns'] / 1e3:.1f} us; "
                     "median (latest) block end of each phase from the first start:")
        lines.append("   " + ", ".join(f"{ph} {v['median_ns'] / 1e3:.1f} ({v['max_ns'] / 1e3:.1f})"
                                       for ph, v in d["phases"].items()))
    for region in REGIONS:
        s = summ.get(region, {"units": 0})
        if not s["units"]:
            lines.append(f" {region}: no routed CTA-pair launch")
            continue
        lines.append(f" {region}: {s['units']} units on CTA 0 ({s['swap_units']} swap), "
                     f"span {s['span_ns'] / 1e3:.1f} us, MMA issue {s['mma_issue_frac']:.2f} "
                     f"and epilogue drain {s['epilogue_drain_frac']:.2f} of it: "
                     f"{s['bound']}-bound")
        for ph, v in s["phases"].items():
            tile = "-" if v["tile_mean_ns"] is None else f"{v['tile_mean_ns'] / 1e3:.2f}"
            sw = "-" if v["swap_mean_ns"] is None else f"{v['swap_mean_ns'] / 1e3:.2f}"
            lines.append(f"   {ph:28s} mean {v['mean_ns'] / 1e3:8.2f} us  total "
                         f"{v['total_ns'] / 1e3:9.1f} us  (pair tiles {tile}, swap units {sw})")
    return "\n".join(lines)


def collect(w, seed: int = 0, warmup: int = 2, device: str = "cuda"):
    """Run `warmup` forward passes of workload `w`, clear the timeline, run
    one more, and return ({region: records}, outputs); the regions are the
    two GEMMs and "dispatch".  Needs the binding to have loaded the timeline
    library (MOE_LIBRARY)."""
    import torch

    from . import binding as B
    from .workloads import make_inputs

    cfg = B.config_of(w)
    inp = make_inputs(w, seed, device)
    a8 = w.acts == "e4m3"
    if w.weights == "e4m3":
        inp = B.quantize_expert_weights(inp, a8=a8)
    outs = B.alloc_outputs(cfg, device, w.D_outer, a8=a8)
    for _ in range(warmup):
        B.forward(cfg, inp, outs)
    torch.cuda.synchronize()
    B.timeline_clear()
    B.forward(cfg, inp, outs)
    torch.cuda.synchronize()
    words = B.timeline_read()
    recs = {region: units(words, i) for i, region in enumerate(REGIONS)}
    recs["dispatch"] = dispatch_blocks(words)
    return recs, outs


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--workload", action="append", required=True,
                    help="a named workload (repeatable)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--json", action="store_true", help="print one JSON line per workload")
    args = ap.parse_args(argv)
    pkg = os.path.dirname(os.path.abspath(__file__))
    os.environ.setdefault("MOE_LIBRARY", os.path.join(pkg, "libmoe_timeline.so"))
    from .workloads import WORKLOADS
    for name in args.workload:
        recs, _ = collect(WORKLOADS[name], seed=args.seed)
        summ = {region: summarize(recs[region]) for region in REGIONS}
        summ["dispatch"] = summarize_dispatch(recs["dispatch"])
        if args.json:
            print(json.dumps({"workload": name, **summ}))
        else:
            print(format_summary(name, summ))
    return 0


if __name__ == "__main__":
    sys.exit(main())
