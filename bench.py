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
DEFAULT_WORKLOAD = "switch_top1_capacity"
L2_FLUSH_BYTES = 512 << 20
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
    """Algorithmic (flops, bytes) of each stage of one forward pass.  With the
    shared expert's tiles inside the routed GEMM launches (shared_fused), the
    routed stages carry the shared work and the shared stages are empty.
    E4M3 expert weights count 1 byte per weight plus a 4-byte scale per row."""
    b = 2 if w.dtype == "bf16" else 4
    D, F, S, T, E, k = w.D, w.F, w.S, w.T, w.E, w.k

    def wbytes(rows, cols):
        return rows * cols + 4 * rows if w.weights == "e4m3" else b * rows * cols

    work = {
        "router": (2 * T * D * E, b * (T * D + E * D) + 4 * T * E),
        "gemm1_routed": (4 * D * F * kept_total,
                         touched * wbytes(2 * F, D) + b * (kept_total * D + kept_total * F)),
        "gemm2_routed": (2 * D * F * kept_total,
                         touched * wbytes(D, F) + b * (kept_total * F + kept_total * D)),
        "gemm1_shared": (4 * D * S * T, wbytes(2 * S, D) + b * (T * D + T * S)),
        "gemm2_shared": (2 * D * S * T, wbytes(D, S) + b * (T * S + T * D)),
        "dispatch": (0, b * (T * D + kept_total * D)),
        "combine": (0, b * (kept_total * D + (T * D if S else 0) + T * D)),
    }
    if shared_fused:
        for r, s in (("gemm1_routed", "gemm1_shared"), ("gemm2_routed", "gemm2_shared")):
            work[r] = (work[r][0] + work[s][0], work[r][1] + work[s][1])
            del work[s]
    return work


def profile_traffic(stage, workload):
    """DRAM bytes per launch of `stage` from a committed ncu summary, if the
    summary was taken on the current source of that stage's kernel (else
    None)."""
    gemm_src = "moe_gemm_w8.cu" if (workload in WORKLOADS and
                                     WORKLOADS[workload].weights == "e4m3" and
                                     stage.startswith("gemm")) else "moe_gemm_tc.cu"
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
def _omp_threads():
    try:
        return int(os.environ.get("OMP_NUM_THREADS", "")) or os.cpu_count()
    except ValueError:
        return os.cpu_count()


def oracle_rate(w, inputs, budget_s=12.0, min_tokens=16):
    """Times the CPU oracle (fp64 loops, OpenMP over tokens) on a bounded
    sample of the workload's tokens.  Returns (tokens/s, sample note)."""
    import oracle  # test infrastructure: only this CPU-baseline leg uses it

    def f32(t):
        return t.detach().float().cpu().numpy()

    T = w.T
    x = inputs["x"]
    b = None if inputs.get("b_r") is None else f32(inputs["b_r"])
    Wr = f32(inputs["W_r"])
    full_weight_bytes = 4 * (3 * w.E * w.D * w.F + 3 * w.D * w.S)
    shared = None
    if w.S:
        shared = (f32(inputs["Ws_gate"]), f32(inputs["Ws_up"]), f32(inputs["Ws_down"]))
    gamma = float(np.float32(w.gamma))

    e4m3 = w.weights == "e4m3"
    if e4m3 and shared is not None:
        # the oracle's own E4M3 codes of the same bf16 weights (untimed)
        shared = tuple(a for W in shared for a in oracle.quantize_e4m3_rows(W))

    def expert(e):
        Ws = (f32(inputs["W_gate"][e]), f32(inputs["W_up"][e]), f32(inputs["W_down"][e]))
        return tuple(a for W in Ws for a in oracle.quantize_e4m3_rows(W)) if e4m3 else Ws

    def rows_fn(xr, ws):
        return oracle.swiglu_rows_q8(xr, *ws) if len(ws) == 6 else oracle.swiglu_rows(xr, *ws)

    if full_weight_bytes <= (6 << 30) and not e4m3:
        Wg, Wu, Wd = f32(inputs["W_gate"]), f32(inputs["W_up"]), f32(inputs["W_down"])
        sh = {} if shared is None else dict(Ws_gate=shared[0], Ws_up=shared[1],
                                            Ws_down=shared[2])

        def run(n):
            xs = f32(x[:n])
            t0 = time.perf_counter()
            oracle.moe_forward(xs, Wr, Wg, Wu, Wd, k=w.k, mode=w.mode, gamma=gamma,
                               alpha=w.alpha, bias=b, bias_selection_only=w.sel_bias, **sh)
            return time.perf_counter() - t0

        n0 = min(T, min_tokens)
        per_tok = run(n0) / n0
        n = int(max(n0, min(T, budget_s / max(per_tok, 1e-9))))
        dt = run(n)
        note = (f"first {n} of {T} tokens: the whole layer (router, gating, capacity over "
                f"the sample, experts, shared expert) in the fp64 oracle")
        return n / dt, note, n

    # weights too large for host memory as fp32: route the sample, then run
    # only the experts it touches, one expert's weights at a time (the
    # device-to-host copies are not timed)
    def run_sampled(n):
        xs = f32(x[:n])
        t0 = time.perf_counter()
        s = oracle.router_logits(xs, Wr, None if w.sel_bias else b)
        idx, wts, _, _ = oracle.route(s, w.k, w.mode, sel_bias=b if w.sel_bias else None)
        dropped, _ = oracle.apply_capacity(idx, w.E, oracle.capacity(n, w.k, w.E, gamma))
        spent = time.perf_counter() - t0
        for e in sorted(set(idx[dropped == 0].ravel().tolist())):
            ws = expert(e)
            rows = np.nonzero(((idx == e) & (dropped == 0)).any(1))[0]
            t0 = time.perf_counter()
            rows_fn(xs[rows], ws)
            spent += time.perf_counter() - t0
        if shared is not None:
            t0 = time.perf_counter()
            rows_fn(xs, shared)
            spent += time.perf_counter() - t0
        return spent

    n = min(T, 8)
    dt = run_sampled(n)
    note = (f"first {n} of {T} tokens: router, gating and capacity over the sample, then each "
            f"touched expert and the shared expert in the fp64 oracle (weight copies"
            f"{' and the oracle E4M3 quantization' if e4m3 else ''} untimed)")
    return n / dt, note, n


# ------------------------------------------------------------------ arms
def workload_config(w, l2_note):
    extra = {"latent_from_d_model": w.D_outer} if w.D_outer else {}
    if w.weights == "e4m3":
        extra["expert_weights"] = "e4m3, one fp32 scale per weight row (bf16 activations)"
    return {**extra, "workload": w.name, "T": w.T, "d_model": w.D, "n_experts": w.E, "d_expert": w.F,
            "top_k": w.k, "d_shared": w.S, "gating": GATING[w.mode],
            "capacity_factor": w.gamma if w.gamma > 0 else None,
            "router_bias": w.bias + (" (selection only)" if w.sel_bias else ""),
            "inputs": "seeded synthetic, resident in HBM", "l2": l2_note}


def run_ours(args, rank, world, device):
    w = WORKLOADS[args.workload]
    torch.cuda.set_device(device)
    cfg = B.config_of(w)
    inputs = make_inputs(w, args.seed + rank, device)
    bf16_inputs = inputs
    if w.weights == "e4m3":
        # the stored weights are E4M3 (quantized once by the library, untimed)
        inputs = B.quantize_expert_weights(bf16_inputs)
    outs = B.alloc_outputs(cfg, device, w.D_outer)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        flush.fill_(1)
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
    for _ in range(args.warmup):
        flush.fill_(1)
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
    for i in range(K):
        flush.fill_(i & 0xFF)                       # evict L2 between steps
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

    # per-stage device time: the instrumented graph, same flush, read per step
    Ks = min(K, 200)
    stage_sum = {n: 0.0 for n in B.STAGES}
    st_s = torch.cuda.Event(enable_timing=True)
    st_e = torch.cuda.Event(enable_timing=True)
    st_total = 0.0
    barrier()
    for i in range(Ks):
        flush.fill_(i & 0xFF)
        st_s.record(stream)
        graph_st.replay()
        st_e.record(stream)
        st_e.synchronize()                          # stage events are re-recorded each replay
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
        flush.fill_(i & 0xFF)
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

    # dominant kernel and its roofline.  Tensor peak: the sustained
    # (power-capped) figure when the kernel runs inside multi-ms steps replayed
    # back to back for at least a second; the burst figure otherwise (short
    # steps, or a timed loop too short for the power cap to act).
    work = stage_work(w, kept_total, touched, B.launch_plan(cfg)["shared_fused"])
    dom = max((n for n in stages if n in work), key=lambda n: stages[n])
    flops, nbytes = work[dom]
    dur_s = stages[dom] / 1e3
    long_steps = ms_per_step >= 1.0 and wall >= 1.0
    tc_peak = peaks["tc_sustained"] if long_steps else peaks["tc"]
    t_tc = flops / (tc_peak * 1e12)
    t_hbm = nbytes / (peaks["hbm"] * 1e9)
    if t_tc >= t_hbm:
        roof = {"bound": "tensor", "achieved": flops / dur_s / 1e12, "peak": tc_peak,
                "unit": "TFLOP/s"}
        roof["frac_of_burst_peak"] = roof["achieved"] / peaks["tc"]
    else:
        roof = {"bound": "hbm", "achieved": nbytes / dur_s / 1e9, "peak": peaks["hbm"],
                "unit": "GB/s"}
        roof["frac_of_8TBs"] = roof["achieved"] / 8000.0
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = profile_traffic(dom, w.name)
    roof["kernel"] = dom
    roof["algorithmic"] = {"flops": flops, "bytes": nbytes}
    roof["avg_launch_ms"] = stages[dom]
    if peaks["source"] != "measured":
        roof["peak_source"] = "fallback"
    elif roof["bound"] == "tensor":
        roof["peak_source"] = ("measured (MEASURED_PEAKS.json bf16_tflops_sustained: multi-ms "
                               "steps back to back for >= 1 s)" if long_steps else
                               "measured (MEASURED_PEAKS.json bf16_tflops burst)")
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
    lt, lbound = RL.roofline_time_s(lf, lb, tc_peak, peaks["hbm"])
    layer = {"bound": lbound, "roofline_ms": lt * 1e3, "frac": lt * 1e3 / ms_per_step,
             "flops": lf, "bytes": lb, "hbm_frac_of_8TBs": lb / (ms_per_step / 1e3) / 8e12}

    # end to end through the C ABI with host buffers (copies inside the timed region)
    x_h = inputs["x"].cpu().pin_memory()
    y_h = torch.empty(outs["y"].shape, dtype=outs["y"].dtype).pin_memory()
    aux_h = torch.empty(1, dtype=torch.float32).pin_memory()
    x_d = torch.empty_like(inputs["x"])
    inp2 = dict(inputs)
    inp2["x"] = x_d
    Ke = min(K, 200)
    e_s = [torch.cuda.Event(enable_timing=True) for _ in range(Ke)]
    e_e = [torch.cuda.Event(enable_timing=True) for _ in range(Ke)]
    barrier()
    for i in range(Ke):
        flush.fill_(i & 0xFF)
        e_s[i].record(stream)
        x_d.copy_(x_h, non_blocking=True)
        B.forward(cfg, inp2, outs)
        y_h.copy_(outs["y"], non_blocking=True)
        aux_h.copy_(outs["aux_loss"], non_blocking=True)
        e_e[i].record(stream)
    barrier()
    e2e_ms = sum(e_s[i].elapsed_time(e_e[i]) for i in range(Ke))
    t = torch.tensor([e2e_ms], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    e2e_value = world * w.T * Ke / (float(t.item()) / 1e3)
    h2d = x_h.numel() * x_h.element_size()
    d2h = y_h.numel() * y_h.element_size() + 4

    # router (unless fused into dispatch), dispatch, GEMM1, GEMM2 (+ two
    # shared-expert GEMMs), combine (unless GEMM2 writes y)
    plan = B.launch_plan(cfg)
    # (with pair tails each routed GEMM is two launches: full 256-row tiles on
    # pairs, segment remainders on single CTAs)
    launches_per_step = (2 if w.D_outer else 0) + \
        (0 if plan["router_fused"] else 1) + 3 + (2 if plan["pair_tails"] else 0) + \
        (2 if w.S and not plan["shared_fused"] else 0) + (0 if plan["direct_y"] else 1)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "step_ms": {"median": statistics.median(step_ms), "min": min(step_ms),
                    "max": max(step_ms), "note": "this rank's CUDA-event time per step"},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": workload_config(w, "flushed between timed steps (512 MiB write)"),
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
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * K,
        "gpu_launches_per_step": launches_per_step,
        "clocks": clk,
        "wall_s_timed_loop": wall,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle  # test infrastructure: only the CPU-baseline leg uses it
        rate, note, n = oracle_rate(w, bf16_inputs, budget_s=args.cpu_budget_s)
        # the same oracle on one host thread (a smaller bounded sample)
        cores = oracle.set_threads(1)
        try:
            rate1, note1, _ = oracle_rate(w, bf16_inputs, budget_s=args.cpu_budget_s / 2,
                                          min_tokens=4)
        finally:
            oracle.set_threads(cores)
        line["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": cores,
                                "kind": "oracle", "sample": note,
                                "single_thread": {"value": rate1, "unit": "tokens/s",
                                                  "cores": 1, "sample": note1}}
    return line


def run_reference(args, world):
    """The CPU oracle as the reference arm (rank 0 only)."""
    w = WORKLOADS[args.workload]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inputs = make_inputs(w, args.seed, dev)
    # each step: the oracle on a bounded token sample, sized so that the
    # whole run stays within ~2 minutes of CPU time
    per_step_budget = max(0.05, 120.0 / max(1, args.steps + args.warmup))
    rate0, note, n = oracle_rate(w, inputs, budget_s=per_step_budget, min_tokens=4)
    times = []
    import oracle

    def f32(t):
        return t.detach().float().cpu().numpy()

    small = 4 * (3 * w.E * w.D * w.F + 3 * w.D * w.S) <= (6 << 30) and w.weights != "e4m3"
    if small:
        args_w = dict(k=w.k, mode=w.mode, gamma=float(np.float32(w.gamma)), alpha=w.alpha,
                      bias=None if inputs.get("b_r") is None else f32(inputs["b_r"]),
                      bias_selection_only=w.sel_bias)
        Wr, Wg, Wu, Wd = (f32(inputs[k]) for k in ("W_r", "W_gate", "W_up", "W_down"))
        sh = {} if not w.S else dict(Ws_gate=f32(inputs["Ws_gate"]), Ws_up=f32(inputs["Ws_up"]),
                                     Ws_down=f32(inputs["Ws_down"]))
        xs = f32(inputs["x"][:n])
        for i in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            oracle.moe_forward(xs, Wr, Wg, Wu, Wd, **args_w, **sh)
            if i >= args.warmup:
                times.append(time.perf_counter() - t0)
        value = n * len(times) / sum(times)
    else:
        value = rate0
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": (sum(times) / len(times) * 1e3) if times else n / value * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, "n/a (host)"),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": _omp_threads(),
                         "kind": "oracle", "sample": note},
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
