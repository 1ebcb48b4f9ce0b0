"""CUDA path vs the CPU oracle, through the C ABI, on seeded inputs.

Small layers span several tiles and ragged tails and are checked on every
token; the benchmark-sized workloads are checked on all routing outputs and
on a seeded sample of y rows, in the launch configuration the benchmark
uses (one moe_forward call on the current stream)."""
import numpy as np
import pytest
import torch

import parity
from mixture_experts_layer_capacity_b300 import binding as B
from mixture_experts_layer_capacity_b300.workloads import WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu

SMALL = [
    # name, T, D, E, F, k, S, mode, gamma, bias
    ("multi_tile_top2", 1000, 256, 8, 384, 2, 192, 0, 0.0, "none"),
    ("ragged_cols_capacity", 777, 192, 16, 320, 4, 0, 1, 0.75, "normal_var2"),
    ("simt_router_e64", 300, 128, 64, 128, 8, 256, 2, 1.0, "none"),
    ("tc_router_e256_zipf", 2048, 512, 256, 128, 8, 0, 2, 0.0, "zipf1.1"),
    ("top1_heavy_drops", 1536, 256, 8, 256, 1, 128, 1, 0.5, "normal_var2"),
    ("k_equals_e", 640, 128, 4, 192, 4, 0, 0, 0.0, "none"),
    ("ragged_chunk_t33", 33, 128, 8, 128, 2, 64, 0, 1.25, "none"),
    # small batch, wide d_model: the router GEMM splits its reduction (fp32
    # partial sums) and the shared expert's tiles run inside the routed GEMMs
    ("split_router_and_shared", 200, 1024, 32, 128, 4, 2048, 2, 0.0, "zipf1.1"),
    # wide down projection (256-column tiles) with fused shared tiles whose
    # rows (T = 300) span three row tiles and whose S is not a multiple of 128
    ("fused_shared_wide_down", 300, 1088, 16, 192, 2, 320, 1, 1.0, "normal_var2"),
]

# Large enough for the CTA-pair GEMMs (>= 16384 rows and >= 512 rows per
# expert), with small D and F so that the oracle stays cheap: y is checked on
# a seeded sample of rows, routing on every token.
PAIR = [
    # ragged segments, partial column tiles (F = 320, D = 192), drops, and
    # a shared expert (dense pair tiles)
    ("pair_ragged_drops", 8200, 192, 4, 320, 2, 256, 1, 0.6, "normal_var2"),
    # one expert per token, no shared expert: the down projection writes y
    ("pair_top1_direct_y", 16400, 256, 8, 256, 1, 0, 2, 1.1, "none"),
    # dropless, several experts empty or tiny, k = 4
    ("pair_dropless_zipf", 4200, 128, 8, 192, 4, 128, 0, 0.0, "zipf1.1"),
    # 128 experts, skewed: many experts under 256 rows run as swap units
    # (narrow down projection: one 64-wide reduction step per swap stage)
    ("pair_tails_e128_zipf", 8200, 128, 128, 192, 8, 0, 2, 0.0, "zipf1.1"),
    # wide down projection (D = 1088 > 1024: 256-column tiles, two reduction
    # steps per swap stage) over F = 320 (five steps: the last stage holds
    # one), partial feature blocks in both GEMMs, small experts as swap units
    ("pair_wide_down_odd_k", 4100, 1088, 16, 320, 4, 0, 2, 0.0, "zipf1.1"),
]


def _w(name, T, D, E, F, k, S, mode, gamma, bias, dtype="bf16", sel_bias=False):
    return Workload(name, T=T, D=D, E=E, F=F, k=k, S=S, mode=mode, gamma=gamma,
                    dtype=dtype, alpha=0.01, bias=bias, sel_bias=sel_bias)


# Sigmoid gating normalised over the chosen experts (mode 3) and a bias that
# only the top-k selection sees, on each router path (fused, tensor-core,
# split tensor-core) and both dtypes: name, T, D, E, F, k, S, mode, gamma,
# bias, sel_bias, dtype
GATING = [
    ("sigmoid_top8_e64", 600, 256, 64, 128, 8, 128, 3, 0.0, "zipf1.1", False, "bf16"),
    ("sigmoid_selbias_e32_drops", 700, 192, 32, 128, 4, 0, 3, 1.0, "normal_var2", True, "bf16"),
    ("softmax_selbias_fused_router", 900, 256, 8, 256, 2, 64, 0, 0.8, "normal_var2", True, "bf16"),
    ("renorm_selbias_split_router", 200, 1024, 64, 128, 8, 0, 2, 0.0, "zipf1.1", True, "bf16"),
    ("raw_top1_selbias", 1024, 128, 16, 128, 1, 0, 1, 1.0, "normal_var2", True, "bf16"),
    ("sigmoid_selbias_fp32", 300, 64, 8, 64, 2, 32, 3, 0.5, "normal_var2", True, "fp32"),
]


# Latent MoE: name, T, L (layer width), E, F, k, S, D_outer, mode, gamma, dtype
LATENT = [
    ("latent_small_bf16", 600, 128, 8, 128, 2, 64, 256, 0, 0.0, "bf16"),
    ("latent_decode_narrow_bf16", 64, 256, 16, 128, 4, 128, 512, 2, 0.0, "bf16"),
    ("latent_capacity_fp32", 200, 64, 4, 64, 2, 32, 96, 1, 0.75, "fp32"),
]


@pytest.mark.parametrize("case", LATENT, ids=[c[0] for c in LATENT])
def test_latent_layers(case):
    name, T, L, E, F, k, S, Do, mode, gamma, dtype = case
    w = Workload(name, T=T, D=L, E=E, F=F, k=k, S=S, mode=mode, gamma=gamma, dtype=dtype,
                 alpha=0.01, D_outer=Do)
    _, inp, outs, code = parity.run(w, seed=14)
    assert code == B.MOE_DEVICE_OK
    assert tuple(outs["y"].shape) == (T, Do)
    print(name, parity.check(w, inp, outs))


@pytest.mark.parametrize("case", GATING, ids=[c[0] for c in GATING])
def test_gating_variants(case):
    name, T, D, E, F, k, S, mode, gamma, bias, sel, dtype = case
    w = _w(name, T, D, E, F, k, S, mode, gamma, bias, dtype=dtype, sel_bias=sel)
    _, inp, outs, code = parity.run(w, seed=12)
    assert code == B.MOE_DEVICE_OK
    rep = parity.check(w, inp, outs)
    if sel:
        # the scores exclude a selection-only bias
        assert "logits_rel" in rep
    print(name, rep)


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    torch.cuda.synchronize()


def test_tiny_fp32_workload():
    w = WORKLOADS["tiny_fp32"]
    _, inp, outs, code = parity.run(w)
    assert code == B.MOE_DEVICE_OK
    rep = parity.check(w, inp, outs)
    assert rep["y_rows"] == w.T


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_bf16_layers(case):
    w = _w(*case)
    _, inp, outs, code = parity.run(w, seed=3)
    assert code == B.MOE_DEVICE_OK
    parity.check(w, inp, outs)


@pytest.mark.parametrize("case", PAIR, ids=[c[0] for c in PAIR])
def test_pair_tile_layers(case):
    w = _w(*case)
    _, inp, outs, code = parity.run(w, seed=6)
    assert code == B.MOE_DEVICE_OK
    rep = parity.check(w, inp, outs, coverage=True, y_sample_n=96)
    print(case[0], rep)


@pytest.mark.parametrize("case", SMALL[:4], ids=[c[0] for c in SMALL[:4]])
def test_small_fp32_layers(case):
    w = _w(*case, dtype="fp32")
    _, inp, outs, code = parity.run(w, seed=4)
    assert code == B.MOE_DEVICE_OK
    parity.check(w, inp, outs)


def test_switch_capacity_workload_every_token():
    w = WORKLOADS["switch_top1_capacity"]
    _, inp, outs, code = parity.run(w)
    assert code == B.MOE_DEVICE_OK
    rep = parity.check(w, inp, outs)
    # the biased router overloads some experts: drops must happen here
    assert int(outs["dropped_mask"].sum()) > 0
    assert int(outs["kept_counts"].max()) == B.capacity(B.config_of(w))
    print(rep)


@pytest.mark.parametrize("name", ["mixtral_decode", "qwen2_57b_decode", "dsv3_decode",
                                  "dsv3_sigmoid_decode", "latent_decode", "latent_prefill",
                                  "mixtral_prefill", "qwen2_57b_prefill", "dsv3_prefill"])
def test_benchmark_sized_workloads_sampled(name):
    """Full-size layers in the benchmark's launch configuration: router
    scores and routing on every token; y on every token of the decode
    layers, and on a coverage sample of at least 512 tokens of the prefill
    layers (every 128-row block of every expert segment, each segment's
    first and last row, every 128-token block of the shared expert)."""
    w = WORKLOADS[name]
    _, inp, outs, code = parity.run(w)
    assert code == B.MOE_DEVICE_OK
    if w.T <= 512:
        rep = parity.check(w, inp, outs)
    else:
        rep = parity.check(w, inp, outs, coverage=True, y_sample_n=512)
        assert rep["y_rows"] >= 512
    print(name, rep)
    del inp, outs
    torch.cuda.empty_cache()


def test_deterministic():
    w = _w(*SMALL[1])
    cfg = B.config_of(w)
    inp = make_inputs(w, 5, "cuda")
    a = B.forward(cfg, inp)
    b = B.forward(cfg, inp)
    for key in ("y", "router_logits", "topk_idx", "topk_w", "dropped_mask",
                "expert_counts", "kept_counts", "aux_loss"):
        assert torch.equal(a[key], b[key]), key


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_single_token(dtype):
    w = _w("one_token", 1, 128, 8, 128, 2, 64, 0, 1.0, "none", dtype=dtype)
    _, inp, outs, code = parity.run(w, seed=8)
    assert code == B.MOE_DEVICE_OK
    parity.check(w, inp, outs)


def test_zero_tokens():
    w = _w("empty", 0, 128, 8, 128, 2, 0, 0, 1.0, "none")
    cfg = B.config_of(w)
    inp = make_inputs(w, 0, "cuda")
    outs = B.alloc_outputs(cfg)
    outs["expert_counts"].fill_(7)
    outs["aux_loss"].fill_(3.0)
    B.forward(cfg, inp, outs)
    torch.cuda.synchronize()
    assert int(outs["expert_counts"].abs().sum()) == 0
    assert float(outs["aux_loss"][0]) == 0.0


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_one_expert_is_the_dense_mlp(mode):
    w = _w("dense", 700, 192, 1, 256, 1, 0, mode, 0.0, "none")
    _, inp, outs, code = parity.run(w, seed=9)
    assert code == B.MOE_DEVICE_OK
    assert torch.all(outs["topk_w"] == 1.0)
    parity.check(w, inp, outs)


def test_nonfinite_input_sets_status():
    w = _w("nan", 64, 64, 4, 64, 2, 0, 0, 0.0, "none", dtype="fp32")
    cfg = B.config_of(w)
    inp = make_inputs(w, 1, "cuda")
    inp["x"][5, 3] = float("nan")
    outs = B.forward(cfg, inp)
    code = B.read_device_status(cfg, outs["workspace"])
    assert code == B.MOE_DEVICE_NONFINITE_SCORE
    idx = outs["topk_idx"].cpu()
    assert int(idx.min()) >= 0 and int(idx.max()) < w.E


def test_runs_on_a_side_stream_and_in_a_cuda_graph():
    w = _w(*SMALL[0])
    cfg = B.config_of(w)
    inp = make_inputs(w, 2, "cuda")
    ref = B.forward(cfg, inp)
    s = torch.cuda.Stream()
    outs = B.alloc_outputs(cfg)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        B.forward(cfg, inp, outs, stream=s)
    s.synchronize()
    assert torch.equal(outs["y"], ref["y"])
    g = torch.cuda.CUDAGraph()
    outs2 = B.alloc_outputs(cfg)
    with torch.cuda.graph(g):
        B.forward(cfg, inp, outs2)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(outs2["y"], ref["y"])
    assert torch.equal(outs2["topk_idx"], ref["topk_idx"])
