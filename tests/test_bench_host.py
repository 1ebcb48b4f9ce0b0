"""Host-side checks of the bench's accounting (no GPU).

The per-stage algorithmic work must add up to the layer's closed forms, a
DRAM-traffic figure from a committed profile summary may only be used while
the kernel source it was taken on is unchanged, and the reference arm (the
oracle on the host) prints its one line on rank 0 only."""
import hashlib
import os
import re

import pytest

import bench
from mixture_experts_layer_capacity_b300 import roofline as RL
from mixture_experts_layer_capacity_b300.workloads import WORKLOADS, Workload

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cases():
    yield Workload("a", T=300, D=128, E=8, F=192, k=2, mode=0, gamma=0.0, dtype="bf16")
    yield Workload("b", T=64, D=256, E=16, F=128, k=4, mode=1, gamma=1.0, dtype="bf16", S=512)
    yield Workload("c", T=96, D=64, E=4, F=128, k=1, mode=2, gamma=0.0, dtype="fp32", S=128)
    yield Workload("d", T=64, D=512, E=32, F=256, k=8, mode=1, gamma=0.0, dtype="bf16",
                   S=256, weights="e4m3")
    yield from WORKLOADS.values()


@pytest.mark.parametrize("w", list(_cases()), ids=lambda w: w.name)
@pytest.mark.parametrize("fused", [False, True])
def test_stage_flops_add_up_to_the_layer(w, fused):
    kept_total, touched = w.T * w.k - 7, min(w.E, 5)
    work = bench.stage_work(w, kept_total, touched, shared_fused=fused and w.S > 0)
    flops = sum(f for f, _ in work.values())
    assert flops == RL.layer_flops(w.T, w.D, w.E, w.F, w.S, kept_total)
    gemm = sum(f for n, (f, _) in work.items() if n.startswith("gemm"))
    assert gemm == RL.expert_flops(w.D, w.F, w.S, w.T, kept_total)


@pytest.mark.parametrize("w", list(_cases()), ids=lambda w: w.name)
@pytest.mark.parametrize("fused", [False, True])
def test_stage_bytes_add_up_to_the_layer(w, fused):
    """The stages' algorithmic bytes add up to the layer's closed form
    (touched expert weights, shared and router weights, x once, y once) and
    the GEMM stages count weights only (no x_perm / h / z traffic)."""
    kept_total, touched = w.T * w.k - 3, min(w.E, 3)
    b = 2 if w.dtype == "bf16" else 4
    work = bench.stage_work(w, kept_total, touched, shared_fused=fused and w.S > 0)
    wb = 1 if w.weights == "e4m3" else None
    layer = RL.layer_bytes(w.T, w.D, w.E, w.F, w.S, touched, b, weight_bytes=wb)
    assert sum(v for _, v in work.values()) == layer
    gemm_bytes = sum(v for n, (_, v) in work.items() if n.startswith("gemm"))
    assert gemm_bytes == layer - b * (w.D * w.E + 2 * w.T * w.D)
    # the GEMM stages' bytes do not grow with the rows they compute
    more = bench.stage_work(w, kept_total + 1000, touched, shared_fused=fused and w.S > 0)
    assert all(more[n][1] == work[n][1] for n in work)


def test_activation_traffic_is_reported_apart():
    w = WORKLOADS["dsv3_prefill"]
    kept = w.T * w.k
    act = bench.stage_activation_bytes(w, kept)
    assert act["gemm1_routed"] == 2 * kept * (w.D + w.F)
    assert act["dispatch"] == 2 * kept * w.D
    fused = bench.stage_activation_bytes(w, kept, shared_fused=True)
    assert "gemm1_shared" not in fused
    assert fused["gemm1_routed"] == act["gemm1_routed"] + act["gemm1_shared"]


def _traffic_lines():
    pat = re.compile(r"bench_traffic:\s*stage=(\S+)\s+workload=(\S+)\s+"
                     r"dram_bytes_per_launch=(\d+)\s+source_sha256=(\w+)")
    pdir = os.path.join(ROOT, "profiles")
    out = []
    for name in sorted(os.listdir(pdir)):
        if name.endswith((".md", ".txt")):
            out += [(name,) + m.groups() for m in pat.finditer(open(os.path.join(pdir, name)).read())]
    return out


def _source_sha(stage, workload):
    if stage in ("dispatch",):
        src = "moe_dispatch.cu"
    elif stage == "combine":
        src = "moe_combine.cu"
    elif stage.startswith("gemm"):
        src = bench.gemm_source(WORKLOADS[workload])
    else:
        src = "moe_gemm_tc.cu"
    path = os.path.join(ROOT, "mixture_experts_layer_capacity_b300", "csrc", src)
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def test_profile_traffic_only_from_current_sources():
    lines = _traffic_lines()
    assert lines, "no bench_traffic lines under profiles/"
    current = 0
    for name, stage, workload, nbytes, sha in lines:
        assert workload in WORKLOADS, (name, workload)
        got = bench.profile_traffic(stage, workload)
        if sha == _source_sha(stage, workload):
            current += 1
            assert got == int(nbytes), (name, stage, workload)
        elif got is not None:
            # another summary holds a current figure for the same stage
            assert any(s == _source_sha(stage, workload) and st == stage and wl == workload
                       for _, st, wl, _, s in lines), (name, stage, workload)
    # the default workload's dominant kernel has a current figure
    assert bench.profile_traffic("gemm1_routed", bench.DEFAULT_WORKLOAD) is not None
    assert current > 0


def test_peaks_are_the_measured_file():
    p = bench._peaks()
    if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")):
        assert p["source"] == "measured"
    assert p["hbm"] > 1000 and p["tc"] > 100 and p["tc_sustained"] <= p["tc"]


def _reference_arm(rank, world):
    import subprocess
    import sys
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--workload", "tiny_fp32", "--steps", "2", "--warmup", "3",
                           "--gpus", str(world)],
                          capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)


def test_reference_arm_prints_one_line_on_rank_zero_only():
    """The reference arm is the oracle on the host; under N ranks only rank 0
    runs it and prints, the others exit 0 without output."""
    import json
    r1 = _reference_arm(1, 2)
    assert r1.returncode == 0, r1.stderr[-2000:]
    assert r1.stdout.strip() == ""
    r0 = _reference_arm(0, 2)
    assert r0.returncode == 0, r0.stderr[-2000:]
    lines = [ln for ln in r0.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 2
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_shared_expert_placement_follows_the_launch_plan():
    """Where the bench books the shared expert's GEMMs: inside the routed
    launches (their stage) or in launches of their own."""
    from mixture_experts_layer_capacity_b300 import binding as B

    def placed(name):
        w = WORKLOADS[name]
        return bench.shared_in_routed(w, B.launch_plan(B.config_of(w)))

    assert not placed("mixtral_decode")            # no shared expert
    assert placed("qwen2_57b_decode")               # bf16, decode: fused tiles
    assert not placed("dsv3_prefill")                # bf16, CTA pairs: own launches
    assert placed("dsv3_decode_fp8")                 # E4M3 weights: always inside
    assert placed("dsv3_decode_w8a8")                # E4M3 activations, few rows
    assert not placed("dsv3_prefill_w8a8")           # E4M3 activations on pairs


def test_e4m3_activation_traffic_counts_the_quantizers():
    w = WORKLOADS["dsv3_prefill_w8a8"]
    kept = w.T * w.k
    act = bench.stage_activation_bytes(w, kept, shared_fused=False)
    bf = bench.stage_activation_bytes(WORKLOADS["dsv3_prefill"], kept, shared_fused=True)
    # the dispatch gathers 1-byte codes and a scale per row instead of bf16 rows
    assert act["dispatch"] == kept * (w.D + 4) < bf["dispatch"]
    # GEMM1 writes fp32 hidden rows and its quantizer reads them back
    assert act["gemm1_routed"] >= kept * 8 * w.F
    # the router stage quantizes every token row once
    assert act["router"] > bf["router"]
