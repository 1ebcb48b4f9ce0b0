#!/usr/bin/env python
"""Benchmark: forward pass of one mixture-of-experts FFN layer on B300 GPUs.

One step = one whole pass of the layer (router, gating, capacity and
dispatch, grouped SwiGLU experts, combine, shared expert, statistics) over
one batch of synthetic tokens, through the C ABI (libmoe.so).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica on its own
batch (weak scaling; the layer needs no exchange between replicas).  Rank 0
prints one JSON line.  `--impl reference` times the CPU oracle as it stands
on the host cores on the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mixture_experts_layer_capacity_b300 import binding as B  # noqa: E402
from mixture_experts_layer_capacity_b300 import roofline as RL  # noqa: E402
from mixture_experts_layer_capacity_b300.workloads import WORKLOADS, make_inputs  # noqa: E402

METRIC = "MoE-layer fwd tokens/s on 1 B300; % of roofline (TC TFLOP/s or HBM GB/s)"
DEFAULT_WORKLOAD = "dsv3_prefill"
L2_FLUSH_BYTES = 512 << 20
L2_BYTES = 126 << 20
GATING = {0: "softmax_over_selected", 1: "softmax_over_all", 2: "softmax_over_all_renormalised",
          3: "sigmoid_normalised_over_selected"}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), tc=float(p["bf16_tflops"]),
                    tc_sustained=float(p["bf16_tflops_sustained"]), source="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm=6400.0, tc=1800.0, tc_sustained=1400.0, source="fallback")


# ------------------------------------------------------------------ clocks
_REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
            0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
            0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
            0x100: "display_clock_setting"}


class _NvmlCtypes:
    """Minimal read-only NVML access through the driver's libnvidia-ml."""

    def __init__(self, uuid):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) != 0:
            raise RuntimeError("nvmlDeviceGetHandleByUUID failed")
        self._reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sm_clock(self):
        v = self.c.c_uint(0)
        self.lib.nvmlDeviceGetClockInfo(self.h, 1, self.c.byref(v))  # NVML_CLOCK_SM
        return int(v.value)

    def max_sm_clock(self):
        v = self.c.c_uint(0)
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, self.c.byref(v))
        return int(v.value)

    def reasons(self):
        v = self.c.c_ulonglong(0)
        self._reasons(self.h, self.c.byref(v))
        return int(v.value)


class ClockSampler:
    """Samples the SM clock and clock-event reasons (read-only NVML) on a
    background thread while the timed region runs."""

    def __init__(self, device, interval_s=0.005):
        self.interval = interval_s
        self.samples, self.reasons = [], 0
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self.nv = None
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            self.nv = _NvmlCtypes(uuid)
            self.max_mhz = self.nv.max_sm_clock()
        except Exception as e:  # noqa: BLE001
            self.err = f"{type(e).__name__}: {e}"

    def _run(self):
        while not self._stop.is_set():
            try:
                self.samples.append(self.nv.sm_clock())
                self.reasons |= self.nv.reasons()
            except Exception:  # noqa: BLE001
                pass
            time.sleep(self.interval)

    def start(self):
        if self.nv is not None:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()

    def stop(self):
        if self._thread is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "note": getattr(self, "err", "nvml unavailable")}
        self._stop.set()
        self._thread.join()
        names = [n for bit, n in _REASONS.items() if self.reasons & bit and bit != 0x1]
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": names,
                "samples": len(self.samples)}


# ------------------------------------------------------------- roofline
def stage_work(w, kept_total, touched, shared_fused=False):
    """Algorithmic (flops, bytes) of each stage of one forward pass, by the
    layer's roofline definition: FLOPs of the kept rows, the shared expert
    and the router; bytes of the touched expert weights, the shared and
    router weights, x read once (counted at the dispatch stage) and y
    written once (combine).  Permutation and intermediate traffic (x_perm,
    h, z) is implementation overhead and is not counted here (see
    stage_activation_bytes).  With the shared expert's tiles inside the
    routed GEMM launches (shared_fused), the routed stages carry the shared
    work and the shared stages are empty.  E4M3 expert weights count 1 byte
    per weight plus a 4-byte scale per row."""
    b = 2 if w.dtype == "bf16" else 4
    D, F, S, T, E, k = w.D, w.F, w.S, w.T, w.E, w.k

    def wbytes(rows, cols):
        if rows * cols == 0:
            return 0
        return rows * cols + 4 * rows if w.weights == "e4m3" else b * rows * cols

    work = {
        "router": (2 * T * D * E, b * E * D),
        "gemm1_routed": (4 * D * F * kept_total, touched * wbytes(2 * F, D)),
        "gemm2_routed": (2 * D * F * kept_total, touched * wbytes(D, F)),
        "gemm1_shared": (4 * D * S * T, wbytes(2 * S, D)),
        "gemm2_shared": (2 * D * S * T, wbytes(D, S)),
        "dispatch": (0, b * T * D),
        "combine": (0, b * T * D),
    }
    if shared_fused:
        for r, s in (("gemm1_routed", "gemm1_shared"), ("gemm2_routed", "gemm2_shared")):
            work[r] = (work[r][0] + work[s][0], work[r][1] + work[s][1])
            del work[s]
    return work


def stage_activation_bytes(w, kept_total, shared_fused=False):
    """Activation bytes each stage moves on top of its algorithmic bytes
    (diagnostic only): the routed GEMMs read x_perm / h and write h / z, the
    shared GEMMs read x / hs and write hs / zs, the dispatch writes x_perm,
    the combine reads z (and zs).  With E4M3 activations the router stage
    also quantizes every token row (reads x, writes codes and scales), the
    dispatch gathers codes and scales instead of bf16 rows, GEMM1 reads
    codes, writes fp32 hidden rows and quantizes them (reads them back,
    writes codes and scales), and GEMM2 reads the hidden codes."""
    b = 2 if w.dtype == "bf16" else 4
    D, F, S, T = w.D, w.F, w.S, w.T
    if w.acts == "e4m3":
        def a8(n, f):   # one row set through GEMM1, the hidden quantizer, GEMM2
            return {"g1": n * (D + 4 + 4 * f + 4 * f + (f + 4)),
                    "g2": n * (f + 4 + b * D)}
        r, sh = a8(kept_total, F), a8(T, S) if S else {"g1": 0, "g2": 0}
        return {"router": b * T * D + 4 * T * w.E + T * (b * D + D + 4),
                "gemm1_routed": r["g1"] + sh["g1"], "gemm2_routed": r["g2"] + sh["g2"],
                "dispatch": kept_total * (D + 4),
                "combine": b * (kept_total * D + (T * D if S else 0))}
    extra = {
        "router": b * T * D + 4 * T * w.E,
        "gemm1_routed": b * kept_total * (D + F),
        "gemm2_routed": b * kept_total * (F + D),
        "gemm1_shared": b * T * (D + S) if S else 0,
        "gemm2_shared": b * T * (S + D) if S else 0,
        "dispatch": b * kept_total * D,
        "combine": b * (kept_total * D + (T * D if S else 0)),
    }
    if shared_fused:
        for r, s in (("gemm1_routed", "gemm1_shared"), ("gemm2_routed", "gemm2_shared")):
            extra[r] += extra.pop(s)
    return extra


def gemm_source(w):
    """The source file of the workload's expert GEMM kernels: the E4M3-weight
    kernels for E4M3 weights with bf16 activations, and for E4M3 activations
    when the layer has few rows per expert (launch plan w8a8_swap); else the
    tile GEMMs."""
    if w.weights != "e4m3":
        return "moe_gemm_tc.cu"
    if w.acts != "e4m3" or B.launch_plan(B.config_of(w))["w8a8_swap"]:
        return "moe_gemm_w8.cu"
    return "moe_gemm_tc.cu"


def shared_in_routed(w, plan):
    """Whether the shared expert's GEMMs run inside the routed GEMM launches
    (as their second problem) rather than in launches of their own: the bf16
    layers by the launch plan, the E4M3-weight layers always, the E4M3-
    activation layers except on CTA pairs."""
    if not w.S:
        return False
    if w.weights != "e4m3":
        return plan["shared_fused"]
    if w.acts == "e4m3":
        return plan["w8a8_swap"] or not plan["pair_routed"]
    return True


def profile_traffic(stage, workload):
    """DRAM bytes per launch of `stage` from a committed ncu summary, if the
    summary was taken on the current source of that stage's kernel (else
    None)."""
    gemm_src = (gemm_source(WORKLOADS[workload]) if workload in WORKLOADS and
                stage.startswith("gemm") else "moe_gemm_tc.cu")
    src_name = {"dispatch": "moe_dispatch.cu", "combine": "moe_combine.cu",
                "router": "moe_gemm_tc.cu"}.get(stage, gemm_src)
    src = os.path.join(ROOT, "mixture_experts_layer_capacity_b300", "csrc", src_name)
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    pat = re.compile(r"bench_traffic:\s*stage=(\S+)\s+workload=(\S+)\s+"
                     r"dram_bytes_per_launch=(\d+)\s+source_sha256=(\w+)")
    pdir = os.path.join(ROOT, "profiles")
    for name in sorted(os.listdir(pdir)) if os.path.isdir(pdir) else []:
        if not name.endswith((".md", ".txt")):
            continue
        for m in pat.finditer(open(os.path.join(pdir, name)).read()):
            if m.group(1) == stage and m.group(2) == workload and m.group(4) == sha:
                return int(m.group(3))
    return None


# ------------------------------------------------------------ CPU oracle
class OracleSample:
    """The CPU oracle (fp64 loops) on a bounded sample of a workload's
    tokens, for the CPU-baseline figures.

    Layers whose weights fit in host memory as fp32 run whole
    (oracle.moe_forward: router, gating, capacity over the sample, experts,
    shared expert; OpenMP over tokens).  Larger layers run the same steps
    expert by expert: the router, gating and capacity over the sample, then
    each expert the sample touches on its rows, then the shared expert.
    Preparation (device-to-host weight copies, the oracle's own E4M3 codes
    for E4M3 workloads) is done once per sample and is not timed."""

    HOST_FP32_LIMIT = 6 << 30

    def __init__(self, w, inputs, n_tokens):
        import oracle  # test infrastructure: only the CPU-baseline legs use it
        self.oracle, self.w = oracle, w
        f32 = self._f32
        self.n = n = max(1, min(w.T, int(n_tokens)))
        self.x = f32(inputs["x"][:n])
        self.b = None if inputs.get("b_r") is None else f32(inputs["b_r"])
        self.Wr = f32(inputs["W_r"])
        self.gamma = float(np.float32(w.gamma))
        self.e4m3 = w.weights == "e4m3"
        self.a8 = w.acts == "e4m3"
        self.whole = self.runs_whole(w)
        q = self._quant
        if self.whole:
            self.W = tuple(f32(inputs[k]) for k in ("W_gate", "W_up", "W_down"))
            self.proj = None if not w.D_outer else (f32(inputs["W_in"]), f32(inputs["W_out"]))
            self.sh = {} if not w.S else {k: f32(inputs[k]) for k in ("Ws_gate", "Ws_up",
                                                                      "Ws_down")}
            return
        self.shared = None
        if w.S:
            self.shared = q(tuple(f32(inputs[k]) for k in ("Ws_gate", "Ws_up", "Ws_down")))
        idx, dropped = self._route()
        self.experts = {}
        for e in sorted(set(idx[dropped == 0].ravel().tolist())):
            self.experts[e] = q(tuple(f32(inputs[k][e]) for k in ("W_gate", "W_up", "W_down")))

    @classmethod
    def runs_whole(cls, w):
        """Whether the sample runs as one oracle.moe_forward call."""
        full_bytes = 4 * (3 * w.E * w.D * w.F + 3 * w.D * w.S)
        return full_bytes <= cls.HOST_FP32_LIMIT and w.weights != "e4m3"

    @staticmethod
    def _f32(t):
        return t.detach().cpu().float().numpy()

    def _quant(self, Ws):
        if not self.e4m3:
            return Ws
        return tuple(a for W in Ws for a in self.oracle.quantize_e4m3_rows(W))

    def _rows(self, xr, ws):
        o = self.oracle
        if len(ws) == 6:
            return (o.swiglu_rows_w8a8 if self.a8 else o.swiglu_rows_q8)(xr, *ws)
        return o.swiglu_rows(xr, *ws)

    def _route(self):
        o, w = self.oracle, self.w
        s = o.router_logits(self.x, self.Wr, None if w.sel_bias else self.b)
        idx, _, _, _ = o.route(s, w.k, w.mode, sel_bias=self.b if w.sel_bias else None)
        dropped, _ = o.apply_capacity(idx, w.E, o.capacity(self.n, w.k, w.E, self.gamma))
        return idx, dropped

    def run(self):
        """One timed pass over the sample; returns seconds."""
        o, w = self.oracle, self.w
        t0 = time.perf_counter()
        if self.whole:
            kw = dict(k=w.k, mode=w.mode, gamma=self.gamma, alpha=w.alpha, bias=self.b,
                      bias_selection_only=w.sel_bias, **self.sh)
            if self.proj is not None:
                o.latent_forward(self.x, *self.proj, self.Wr, *self.W, **kw)
            else:
                o.moe_forward(self.x, self.Wr, *self.W, **kw)
            return time.perf_counter() - t0
        idx, dropped = self._route()
        for e, ws in self.experts.items():
            rows = np.nonzero(((idx == e) & (dropped == 0)).any(1))[0]
            if rows.size:
                self._rows(self.x[rows], ws)
        if self.shared is not None:
            self._rows(self.x, self.shared)
        return time.perf_counter() - t0

    def note(self):
        w = self.w
        if self.whole:
            what = "the whole latent layer (projections, " if w.D_outer else "the whole layer ("
            return (f"first {self.n} of {w.T} tokens: {what}router, gating, capacity "
                    f"over the sample, experts, shared expert) in the fp64 oracle")
        return (f"first {self.n} of {w.T} tokens: router, gating and capacity over the sample, "
                f"then each of the {len(self.experts)} experts it touches on its rows and the "
                f"shared expert, in the fp64 oracle (weight copies"
                f"{' and the oracle E4M3 quantization' if self.e4m3 else ''} untimed"
                f"{'; token and hidden rows quantized to E4M3 inside the timed oracle' if self.a8 else ''})")


SAMPLED_TOKENS = 8   # tokens of an expert-by-expert sample (bounds its host weight copies)


def oracle_rate(w, inputs, budget_s=12.0, n0=8):
    """Times the CPU oracle on a bounded sample taking about budget_s.  A
    whole small layer: a probe on n0 tokens sizes the sample.  A large layer
    (expert by expert): SAMPLED_TOKENS tokens, timed as many times as fit in
    the budget.  Returns (tokens/s, note)."""
    if OracleSample.runs_whole(w):
        probe = OracleSample(w, inputs, n0)
        per_tok = probe.run() / probe.n
        n = int(max(probe.n, min(w.T, budget_s / max(per_tok, 1e-9))))
        if n != probe.n:
            del probe
            smp = OracleSample(w, inputs, n)
        else:
            smp = probe
        return smp.n / smp.run(), smp.note()
    smp = OracleSample(w, inputs, SAMPLED_TOKENS)
    total, reps = 0.0, 0
    while reps == 0 or (total < budget_s and reps < 50):
        total += smp.run()
        reps += 1
    return smp.n * reps / total, smp.note() + f", timed {reps} times"


# ------------------------------------------------------------------ arms
def workload_config(w):
    extra = {"latent_from_d_model": w.D_outer} if w.D_outer else {}
    if w.weights == "e4m3" and w.acts == "e4m3":
        extra["expert_weights"] = "e4m3, one fp32 scale per weight row"
        extra["expert_activations"] = ("e4m3, one fp32 scale per token row and per hidden row "
                                       "(quantized inside the layer)")
    elif w.weights == "e4m3":
        extra["expert_weights"] = "e4m3, one fp32 scale per weight row (bf16 activations)"
    return {**extra, "workload": w.name, "T": w.T, "d_model": w.D, "n_experts": w.E, "d_expert": w.F,
            "top_k": w.k, "d_shared": w.S, "gating": GATING[w.mode],
            "capacity_factor": w.gamma if w.gamma > 0 else None,
            "router_bias": w.bias + (" (selection only)" if w.sel_bias else ""),
            "inputs": "seeded synthetic, resident in HBM"}


class nvtx_range:
    """An NVTX range around a phase of the bench (seen by nsys or ncu's
    NVTX filters; a no-op when no profiler is attached)."""

    def __init__(self, name):
        self.name = name

    def __enter__(self):
        try:
            torch.cuda.nvtx.range_push(self.name)
            self.pushed = True
        except Exception:   # NVTX unavailable in this build
            self.pushed = False
        return self

    def __exit__(self, *exc):
        if self.pushed:
            torch.cuda.nvtx.range_pop()
        return False


def run_ours(args, rank, world, device):
    w = WORKLOADS[args.workload]
    torch.cuda.set_device(device)
    cfg = B.config_of(w)
    inputs = make_inputs(w, args.seed + rank, device)
    bf16_inputs = inputs
    if w.weights == "e4m3":
        # the stored weights are E4M3 (quantized once by the library, untimed)
        inputs = B.quantize_expert_weights(bf16_inputs, a8=w.acts == "e4m3")
    outs = B.alloc_outputs(cfg, device, w.D_outer, a8=w.acts == "e4m3")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()
    # L2 between steps: a layer whose inputs (weights, x) exceed twice the L2
    # streams them through it every step, so no step finds the previous
    # one's data there and no flush is needed; smaller layers get a 512 MiB
    # write before every step (outside the timed events; the write-back of
    # its dirty lines lands inside the next step).
    input_bytes = sum(v.numel() * v.element_size() for v in inputs.values()
                      if isinstance(v, torch.Tensor))
    big_inputs = input_bytes > 2 * L2_BYTES

    def evict(i):
        if not big_inputs:
            flush.fill_(i & 0xFF)

    for i in range(args.warmup):
        evict(i)
        B.forward(cfg, inputs, outs)
    torch.cuda.synchronize()
    code = B.read_device_status(cfg, outs["workspace"])
    if code != B.MOE_DEVICE_OK:
        raise RuntimeError(f"device status {code} after warm-up")

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    # The timed step replays one moe_forward captured in a CUDA graph.  A
    # second graph of the same call carries the library's stage events (each
    # event node costs ~1 us and breaks launch overlap, so it is timed in a
    # separate pass and gives the per-kernel durations).
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        B.forward(cfg, inputs, outs)
    stage_ev = B.StageEvents()
    graph_st = torch.cuda.CUDAGraph()
    with stage_ev:
        with torch.cuda.graph(graph_st):
            B.forward(cfg, inputs, outs)
    for i in range(args.warmup):
        evict(i)
        graph.replay()
        graph_st.replay()
    torch.cuda.synchronize()

    K = args.steps
    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    clocks = ClockSampler(device)
    barrier()
    clocks.start()
    wall0 = time.perf_counter()
    with nvtx_range("moe timed steps"):
        for i in range(K):
            evict(i)                                # L2 between steps (above)
            ev_s[i].record(stream)
            graph.replay()
            ev_e[i].record(stream)
        barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()

    step_ms = [ev_s[i].elapsed_time(ev_e[i]) for i in range(K)]
    total_ms = sum(step_ms)
    t = torch.tensor([total_ms], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    total_ms_max = float(t.item())
    ms_per_step = total_ms_max / K
    value = world * w.T * K / (total_ms_max / 1e3)
    code = B.read_device_status(cfg, outs["workspace"])
    if code != B.MOE_DEVICE_OK:
        raise RuntimeError(f"device status {code} after the timed steps")

    # per-stage device time: the instrumented graph, same L2 policy, read per step
    Ks = min(K, 200)
    stage_sum = {n: 0.0 for n in B.STAGES}
    st_s = torch.cuda.Event(enable_timing=True)
    st_e = torch.cuda.Event(enable_timing=True)
    st_total = 0.0
    barrier()
    with nvtx_range("moe instrumented steps"):
        for i in range(Ks):
            evict(i)
            st_s.record(stream)
            graph_st.replay()
            st_e.record(stream)
            st_e.synchronize()                      # stage events are re-recorded each replay
            st_total += st_s.elapsed_time(st_e)
            for n, v in stage_ev.elapsed_ms().items():
                stage_sum[n] += v
    stages = {n: v / Ks for n, v in stage_sum.items()}
    staged_ms = st_total / Ks

    # the same steps as direct moe_forward calls (no graph), for reference
    Kq = min(K, 200)
    q_s = [torch.cuda.Event(enable_timing=True) for _ in range(Kq)]
    q_e = [torch.cuda.Event(enable_timing=True) for _ in range(Kq)]
    barrier()
    for i in range(Kq):
        evict(i)
        q_s[i].record(stream)
        B.forward(cfg, inputs, outs)
        q_e[i].record(stream)
    barrier()
    eager_ms = sum(q_s[i].elapsed_time(q_e[i]) for i in range(Kq)) / Kq

    kept = outs["kept_counts"].cpu().numpy()
    counts = outs["expert_counts"].cpu().numpy()
    kept_total = int(kept.sum())
    touched = int((kept > 0).sum())
    peaks = _peaks()

    # dominant kernel and its roofline: the algorithmic work of the stage
    # (FLOPs of the kept rows; touched weight bytes) against the measured
    # peaks.  The timed loop replays the layer back to back, but at the
    # default step count it lasts well under a second, so the tensor figure
    # is held to the burst peak; the fraction of the sustained (power-capped)
    # peak is reported beside it.
    fused = shared_in_routed(w, B.launch_plan(cfg))
    work = stage_work(w, kept_total, touched, fused)
    act = stage_activation_bytes(w, kept_total, fused)
    dom = max((n for n in stages if n in work), key=lambda n: stages[n])
    flops, nbytes = work[dom]
    dur_s = stages[dom] / 1e3
    # E4M3 x E4M3 GEMMs: the measured bf16 peak times the nominal dense
    # E4M3 : bf16 ratio (4.5 : 2.25 PFLOP/s)
    a8 = w.acts == "e4m3"
    fp8_ratio = 2.0
    tc_peak = peaks["tc"] * (fp8_ratio if a8 and dom.startswith("gemm") else 1.0)
    tc_sus = peaks["tc_sustained"] * (fp8_ratio if a8 and dom.startswith("gemm") else 1.0)
    t_tc = flops / (tc_peak * 1e12)
    t_hbm = nbytes / (peaks["hbm"] * 1e9)
    if t_tc >= t_hbm:
        roof = {"bound": "tensor", "achieved": flops / dur_s / 1e12, "peak": tc_peak,
                "unit": "TFLOP/s"}
        roof["frac_of_sustained_peak"] = roof["achieved"] / tc_sus
    else:
        roof = {"bound": "hbm", "achieved": nbytes / dur_s / 1e9, "peak": peaks["hbm"],
                "unit": "GB/s"}
        roof["frac_of_8TBs"] = roof["achieved"] / 8000.0
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = profile_traffic(dom, w.name)
    roof["kernel"] = dom
    roof["algorithmic"] = {"flops": flops, "bytes": nbytes,
                           "note": "FLOPs of the kept rows (no padding); bytes of the touched "
                                   "weights; x_perm/h/z traffic excluded"}
    roof["bytes_with_activations"] = nbytes + act[dom]
    roof["avg_launch_ms"] = stages[dom]
    if peaks["source"] != "measured":
        roof["peak_source"] = "fallback"
    elif roof["bound"] == "tensor" and tc_peak != peaks["tc"]:
        roof["peak_source"] = ("measured bf16 burst (MEASURED_PEAKS.json bf16_tflops) x 2, "
                               "the nominal dense E4M3 : bf16 ratio")
    elif roof["bound"] == "tensor":
        roof["peak_source"] = "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    else:
        roof["peak_source"] = "measured (MEASURED_PEAKS.json hbm_gbs)"

    # whole-layer roofline (slower of algorithmic FLOPs at TC peak and bytes at HBM)
    lf = RL.layer_flops(w.T, w.D, w.E, w.F, w.S, kept_total)
    lb = RL.layer_bytes(w.T, w.D, w.E, w.F, w.S, touched, 2 if w.dtype == "bf16" else 4,
                        weight_bytes=1 if w.weights == "e4m3" else None)
    if w.D_outer:
        # the latent layer's two projections: 2*T*D_outer*D FLOPs and D_outer*D
        # weights each; x and y at the outer width instead of the latent one
        esz = 2 if w.dtype == "bf16" else 4
        lf += 4 * w.T * w.D_outer * w.D
        lb += esz * (2 * w.D_outer * w.D + 2 * w.T * (w.D_outer - w.D))
    # the layer's tensor time: E4M3 expert GEMMs at twice the bf16 rate
    ef = RL.expert_flops(w.D, w.F, w.S, w.T, kept_total) if a8 else 0
    lf_bf16 = lf - ef + ef / fp8_ratio          # bf16-equivalent FLOPs
    lt, lbound = RL.roofline_time_s(lf_bf16, lb, peaks["tc"], peaks["hbm"])
    layer = {"bound": lbound, "roofline_ms": lt * 1e3, "frac": lt * 1e3 / ms_per_step,
             "flops": lf, "bytes": lb, "hbm_frac_of_8TBs": lb / (ms_per_step / 1e3) / 8e12}
    if a8:
        layer["note"] = "expert GEMM FLOPs at 2x the measured bf16 peak (E4M3 operands)"
    if lbound == "tensor":
        layer["frac_of_sustained_peak"] = (lf_bf16 / (peaks["tc_sustained"] * 1e12)) / (ms_per_step / 1e3)

    # end to end through the C ABI with host buffers: every step copies its
    # x from pinned host memory to the device, runs moe_forward and reads y
    # and the balance loss back into pinned host memory, all inside the timed
    # region.  Three streams (upload, compute, download) and two buffer slots
    # let step i+1's upload and step i-1's download overlap step i's compute;
    # events order each slot's reuse.  Workloads whose inputs exceed twice
    # the L2 need no flush between steps; smaller ones flush L2 on the
    # compute stream before every step (its time is then part of e2e).
    x_h = inputs["x"].cpu().pin_memory()
    slots = []
    for _ in range(2):
        o = dict(outs)
        o["y"] = torch.empty_like(outs["y"])
        o["aux_loss"] = torch.empty_like(outs["aux_loss"])
        inp_s = dict(inputs)
        inp_s["x"] = torch.empty_like(inputs["x"])
        slots.append(dict(inp=inp_s, outs=o,
                          y_h=torch.empty(o["y"].shape, dtype=o["y"].dtype).pin_memory(),
                          aux_h=torch.empty(1, dtype=torch.float32).pin_memory(),
                          up=torch.cuda.Event(), comp=torch.cuda.Event(),
                          down=torch.cuda.Event()))
    s_up, s_down = torch.cuda.Stream(device), torch.cuda.Stream(device)
    Ke = min(K, 200)

    def e2e_steps(n):
        for i in range(n):
            sl = slots[i % 2]
            if i >= 2:
                s_up.wait_event(sl["comp"])      # compute i-2 has read this slot's x
            with torch.cuda.stream(s_up):
                sl["inp"]["x"].copy_(x_h, non_blocking=True)
            sl["up"].record(s_up)
            stream.wait_event(sl["up"])
            if i >= 2:
                stream.wait_event(sl["down"])    # download i-2 has read this slot's y
            evict(i)
            B.forward(cfg, sl["inp"], sl["outs"], stream=stream)
            sl["comp"].record(stream)
            s_down.wait_event(sl["comp"])
            with torch.cuda.stream(s_down):
                sl["y_h"].copy_(sl["outs"]["y"], non_blocking=True)
                sl["aux_h"].copy_(sl["outs"]["aux_loss"], non_blocking=True)
            sl["down"].record(s_down)
        for sl in slots:
            stream.wait_event(sl["down"])

    e2e_steps(2)                                   # warm the copy paths
    barrier()
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    s_up.wait_stream(stream)
    with nvtx_range("moe end-to-end steps"):
        e2e_steps(Ke)
    e_end.record(stream)
    barrier()
    t = torch.tensor([e_start.elapsed_time(e_end)], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    e2e_value = world * w.T * Ke / (float(t.item()) / 1e3)
    h2d = x_h.numel() * x_h.element_size()
    d2h = slots[0]["y_h"].numel() * slots[0]["y_h"].element_size() + 4
    # the copy rates alone (one upload, one download, nothing else running)
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    rates = {}
    for name, dst, srcb, nb in (("h2d_gbs", slots[0]["inp"]["x"], x_h, h2d),
                                ("d2h_gbs", slots[0]["y_h"], slots[0]["outs"]["y"], d2h - 4)):
        best = float("inf")
        for _ in range(3):
            c0.record(stream)
            dst.copy_(srcb, non_blocking=True)
            c1.record(stream)
            c1.synchronize()
            best = min(best, c0.elapsed_time(c1))
        rates[name] = nb / (best / 1e3) / 1e9

    # router (unless fused into dispatch), dispatch, GEMM1, GEMM2 (+ two
    # shared-expert GEMMs), combine (unless GEMM2 writes y); a latent layer
    # adds its two projections
    # with E4M3 activations the token rows (once per token) and the hidden
    # rows (routed, shared) are quantized by one launch each
    plan = B.launch_plan(cfg)
    shared_apart = w.S and not shared_in_routed(w, plan)
    launches_per_step = (2 if w.D_outer else 0) + \
        (0 if plan["router_fused"] else 1) + 3 + \
        (2 if shared_apart else 0) + (0 if plan["direct_y"] else 1) + \
        ((2 + (1 if w.S else 0)) if a8 else 0)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "step_ms": {"median": statistics.median(step_ms), "min": min(step_ms),
                    "max": max(step_ms), "note": "this rank's CUDA-event time per step"},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3" if a8 else ("bf16" if w.dtype == "bf16" else "f32"),
        "data": "synthetic",
        "config": workload_config(w),
        "l2": (f"inputs larger than L2 ({input_bytes / 2**30:.2f} GiB of weights and x), "
               "no flush between timed steps" if big_inputs else
               "flushed between timed steps (512 MiB write)"),
        "launch": "one moe_forward captured in a CUDA graph, replayed per step",
        "eager": {"value": world * w.T / (eager_ms / 1e3), "ms_per_step": eager_ms,
                  "note": "direct moe_forward calls, no graph"},
        "instrumented_ms_per_step": staged_ms,
        "roofline": roof,
        "layer_roofline": layer,
        "stages_ms": stages,
        "routing": {"kept_total": kept_total, "touched_experts": touched,
                    "busiest_share": float(counts.max() / max(1, counts.sum())),
                    "drop_fraction": float(1.0 - kept_total / max(1, w.T * w.k))},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": Ke, **rates,
                "note": "pinned host x uploaded and y + balance loss downloaded every step; "
                        "uploads, compute and downloads on three streams, two buffer slots; "
                        + ("inputs larger than L2, no flush" if big_inputs else
                           "L2 flushed on the compute stream before every step")},
        "gpu_launches": launches_per_step * K,
        "gpu_launches_per_step": launches_per_step,
        "clocks": clk,
        "wall_s_timed_loop": wall,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle  # test infrastructure: only the CPU-baseline leg uses it
        # whole small layers spread their tokens over all host threads; the
        # expert-by-expert sample of a large layer gives each expert only a
        # few rows to spread, so it is timed on one thread
        whole = OracleSample.runs_whole(w)
        cores = (os.cpu_count() or 1) if whole else 1
        threads = oracle.set_threads(cores)
        try:
            rate, note = oracle_rate(w, bf16_inputs, budget_s=args.cpu_budget_s)
        finally:
            oracle.set_threads(threads)
        line["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": cores,
                                "kind": "oracle", "sample": note}
    return line


def run_reference(args, world):
    """The CPU oracle as the reference arm (rank 0 only): every step runs the
    oracle on the same bounded token sample of the workload, sized so that
    the whole run stays within about two minutes of CPU time."""
    import oracle  # test infrastructure: the reference arm is the oracle
    w = WORKLOADS[args.workload]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inputs = make_inputs(w, args.seed, dev)
    whole = OracleSample.runs_whole(w)
    cores = (os.cpu_count() or 1) if whole else 1
    threads = oracle.set_threads(cores)
    try:
        per_step_budget = max(0.05, 120.0 / max(1, args.steps + args.warmup))
        probe = OracleSample(w, inputs, 16 if whole else 4)
        per_tok = probe.run() / probe.n
        n = int(max(1, min(w.T, per_step_budget / max(per_tok, 1e-9))))
        if not whole:
            n = min(n, SAMPLED_TOKENS)   # bounds the untimed host weight copies
        if n != probe.n:
            del probe
            smp = OracleSample(w, inputs, n)
        else:
            smp = probe
        times = [smp.run() for _ in range(args.warmup + args.steps)][args.warmup:]
    finally:
        oracle.set_threads(threads)
    value = smp.n * len(times) / sum(times)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sum(times) / len(times) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                         "kind": "oracle", "sample": smp.note() + " per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, world)), flush=True)
        return

    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local)
    line = run_ours(args, rank, world, device)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
