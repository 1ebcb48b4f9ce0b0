"""E4M3 activations as well as E4M3 expert weights (moe_forward_w8a8)
against the CPU oracle, through the C ABI.

The quantized activations the library leaves in its workspace are checked
bit for bit: the permuted token rows' codes and scales against the oracle's
row quantizer applied to the same token rows in expert order, and the hidden
rows' codes and scales against the oracle's quantizer applied to the
library's own fp32 hidden rows (the hidden values themselves come out of a
GPU reduction whose rounding order differs from the oracle's, so they are
compared within tolerance through y).  Routing is checked as for bf16
weights and y against the oracle's fp64 layer with quantized activations
(oracle.swiglu_rows_w8a8), at the bf16 tolerance."""
import numpy as np
import pytest
import torch

import oracle
import parity
from mixture_experts_layer_capacity_b300 import binding as B
from mixture_experts_layer_capacity_b300.workloads import WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    torch.cuda.synchronize()


def _expert_order(idx, dropped, E):
    """Token of each kept assignment in the layer's expert order (experts
    ascending, tokens ascending within an expert)."""
    T, k = idx.shape
    t_all = np.repeat(np.arange(T), k)
    e_all = idx.ravel().astype(np.int64)
    kept = dropped.ravel() == 0
    t_k, e_k = t_all[kept], e_all[kept]
    return t_k[np.lexsort((t_k, e_k))]


def _check_quantized_rows(w, inp, outs, max_rows=None):
    """Bit-exact checks of the quantized token and hidden rows: all of them,
    or (max_rows) the first, the last and a seeded sample."""
    cfg = B.config_of(w)
    idx = outs["topk_idx"].cpu().numpy()
    dropped = outs["dropped_mask"].cpu().numpy()
    order = _expert_order(idx, dropped, w.E)
    R = int(outs["kept_counts"].sum())
    assert order.size == R
    rows = np.arange(R)
    if max_rows is not None and R > max_rows:
        rng = np.random.default_rng(3)
        rows = np.unique(np.concatenate([[0, R - 1], rng.choice(R, max_rows, replace=False)]))
    sel = torch.as_tensor(rows, device=inp["x"].device)
    act = B.w8a8_activations(cfg, outs["workspace"], R)
    x = parity.f32(inp["x"])
    q_ref, s_ref = oracle.quantize_e4m3_rows(x[order[rows]])
    np.testing.assert_array_equal(act["x_scales"][sel].cpu().numpy(), s_ref)
    np.testing.assert_array_equal(act["x_codes"][sel].cpu().numpy(), q_ref)
    h = act["h_values"][sel].cpu().numpy()
    assert np.isfinite(h).all()
    hq_ref, hs_ref = oracle.quantize_e4m3_rows(h)
    np.testing.assert_array_equal(act["h_scales"][sel].cpu().numpy(), hs_ref)
    np.testing.assert_array_equal(act["h_codes"][sel].cpu().numpy(), hq_ref)
    return R


# name, T, D, E, F, k, S, mode, gamma, bias.  Layers with at most 64 rows per
# expert on average run the weights-as-M-operand kernels (launch plan
# w8a8_swap: 32-row token units), the others 128-row token tiles.
CASES = [
    # tiles: shared expert narrower than the routed ones; several token tiles
    ("a8_multi_tile_top2", 1000, 256, 8, 384, 2, 192, 0, 0.0, "none"),
    # tiles: F = 320 and D = 192 leave partial tiles and a half-empty last
    # 128-wide reduction step; capacity drops
    ("a8_ragged_capacity_e16", 777, 192, 16, 320, 4, 0, 1, 0.75, "normal_var2"),
    # tiles: segments of ~250 rows, several 128-row tiles per expert
    ("a8_long_segments", 500, 128, 4, 128, 2, 0, 0, 0.0, "none"),
    # swap: decode-like, 64 experts, shared down projection cut into
    # S / F = 8 pieces
    ("a8_decode_e64_shared_pieces", 64, 512, 64, 128, 8, 1024, 2, 0.0, "zipf1.1"),
    # swap: k = 1 without a shared expert, the down projection writes y
    ("a8_top1_direct_y", 300, 256, 8, 256, 1, 0, 1, 1.0, "normal_var2"),
    # swap: one token, wide d_model (256-feature units, a ragged one)
    ("a8_one_token_wide", 1, 1088, 8, 192, 2, 320, 0, 0.0, "none"),
    # swap: d_expert = 64 without a shared expert (a half-filled reduction step)
    ("a8_narrow_expert", 200, 256, 8, 64, 2, 0, 0, 0.0, "none"),
    # swap: ragged features and d_model with capacity drops; segments of
    # 30-70 rows (one or two 32-row units, 16-row MMAs for the rest)
    ("a8_swap_capacity_e16", 200, 192, 16, 320, 4, 0, 1, 0.75, "normal_var2"),
    # swap: wide d_model, shared expert wider than the routed ones (two
    # pieces of its down projection)
    ("a8_swap_shared_wide", 40, 1088, 8, 256, 2, 384, 0, 0.0, "none"),
]


# Large enough for the CTA-pair GEMMs (>= 16384 routed rows, >= 512 per
# expert): 256-row pair tiles, experts under 256 rows as swap units, the
# shared expert's dense pair tiles; small D and F keep the oracle cheap.
PAIR = [
    # ragged segments, partial column tiles (F = 320, D = 192), drops, and
    # a shared expert (dense pair tiles)
    ("a8_pair_ragged_drops", 8200, 192, 4, 320, 2, 256, 1, 0.6, "normal_var2"),
    # one expert per token, no shared expert: the down projection writes y
    ("a8_pair_top1_direct_y", 16400, 256, 8, 256, 1, 0, 2, 1.1, "none"),
    # 128 experts, skewed: many experts under 256 rows run as swap units
    ("a8_pair_tails_e128_zipf", 8200, 128, 128, 192, 8, 0, 2, 0.0, "zipf1.1"),
    # wide down projection (256-column tiles, two reduction steps per swap
    # stage) over F = 320 (three 128-wide steps, the last half empty)
    ("a8_pair_wide_down_odd_k", 4100, 1088, 16, 320, 4, 0, 2, 0.0, "zipf1.1"),
]


@pytest.mark.parametrize("case", PAIR, ids=[c[0] for c in PAIR])
def test_w8a8_pair_layers(case):
    name, T, D, E, F, k, S, mode, gamma, bias = case
    w = Workload(name, T=T, D=D, E=E, F=F, k=k, S=S, mode=mode, gamma=gamma, dtype="bf16",
                 alpha=0.01, bias=bias, weights="e4m3", acts="e4m3")
    assert B.launch_plan(B.config_of(w))["pair_routed"]
    _, inp, outs, code = parity.run(w, seed=29)
    assert code == B.MOE_DEVICE_OK
    R = _check_quantized_rows(w, inp, outs, max_rows=4096)
    rep = parity.check(w, inp, outs, e4m3=True, a8=True, coverage=True, y_sample_n=96)
    rep["rows"] = R
    print(name, rep)


def test_cases_cover_both_kernel_forms():
    forms = {B.launch_plan(B.make_config(T, D, E, F, k, d_shared=S))["w8a8_swap"]
             for _, T, D, E, F, k, S, *_ in CASES}
    assert forms == {True, False}


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_w8a8_layers(case):
    name, T, D, E, F, k, S, mode, gamma, bias = case
    w = Workload(name, T=T, D=D, E=E, F=F, k=k, S=S, mode=mode, gamma=gamma, dtype="bf16",
                 alpha=0.01, bias=bias, weights="e4m3", acts="e4m3")
    _, inp, outs, code = parity.run(w, seed=23)
    assert code == B.MOE_DEVICE_OK
    R = _check_quantized_rows(w, inp, outs)
    rep = parity.check(w, inp, outs, e4m3=True, a8=True)
    rep["rows"] = R
    print(name, rep)


def test_w8a8_zero_tokens():
    w = Workload("a8_empty", T=0, D=128, E=8, F=128, k=2, S=128, mode=0, gamma=1.0,
                 weights="e4m3", acts="e4m3")
    cfg = B.config_of(w)
    inp = B.quantize_expert_weights(make_inputs(w, 0, "cuda"), a8=True)
    outs = B.alloc_outputs(cfg, a8=True)
    outs["expert_counts"].fill_(7)
    outs["aux_loss"].fill_(3.0)
    B.forward(cfg, inp, outs)
    torch.cuda.synchronize()
    assert int(outs["expert_counts"].abs().sum()) == 0
    assert float(outs["aux_loss"][0]) == 0.0


def test_w8a8_rejects_the_bf16_workspace():
    w = Workload("a8_ws", T=32, D=128, E=4, F=128, k=2, weights="e4m3", acts="e4m3")
    cfg = B.config_of(w)
    inp = B.quantize_expert_weights(make_inputs(w, 0, "cuda"), a8=True)
    outs = B.alloc_outputs(cfg)                  # sized for moe_forward
    with pytest.raises(B.MoeError) as ei:
        B.forward(cfg, inp, outs)
    assert ei.value.status == B.MOE_ERR_WORKSPACE


@pytest.mark.parametrize("name", ["mixtral_decode_w8a8", "qwen2_57b_decode_w8a8",
                                  "dsv3_decode_w8a8"])
def test_w8a8_benchmark_sized_decode(name):
    w = WORKLOADS[name]
    _, inp, outs, code = parity.run(w)
    assert code == B.MOE_DEVICE_OK
    _check_quantized_rows(w, inp, outs)
    # decode-sized: scores, routing and y on every token
    rep = parity.check(w, inp, outs, e4m3=True, a8=True)
    assert rep["y_rows"] == w.T
    print(name, rep)
    del inp, outs
    torch.cuda.empty_cache()


def test_w8a8_benchmark_sized_prefill():
    w = WORKLOADS["dsv3_prefill_w8a8"]
    _, inp, outs, code = parity.run(w)
    assert code == B.MOE_DEVICE_OK
    _check_quantized_rows(w, inp, outs, max_rows=8192)
    rep = parity.check(w, inp, outs, e4m3=True, a8=True, coverage=True, y_sample_n=256,
                       logit_rows=np.arange(w.T))
    print(w.name, rep)
    del inp, outs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("case", [CASES[0], CASES[3], PAIR[0]], ids=lambda c: c[0])
def test_w8a8_runs_are_bit_identical(case):
    """No float atomics and fixed reduction orders: two calls on the same
    inputs give the same bits (tile, weights-as-M and CTA-pair forms)."""
    name, T, D, E, F, k, S, mode, gamma, bias = case
    w = Workload(name, T=T, D=D, E=E, F=F, k=k, S=S, mode=mode, gamma=gamma, dtype="bf16",
                 alpha=0.01, bias=bias, weights="e4m3", acts="e4m3")
    cfg = B.config_of(w)
    inp = B.quantize_expert_weights(make_inputs(w, 37, "cuda"), a8=True)
    a = B.forward(cfg, inp)
    b = B.forward(cfg, inp)
    torch.cuda.synchronize()
    for key in ("y", "router_logits", "topk_idx", "topk_w", "dropped_mask", "expert_counts",
                "kept_counts", "aux_loss"):
        assert torch.equal(a[key], b[key]), key


@pytest.mark.parametrize("rows", [200, 9000], ids=["swap_form", "pair_form"])
def test_w8a8_sigmoid_gating_with_selection_bias(rows):
    """DeepSeek-V3's own gating (sigmoid scores normalised over the chosen
    experts, a bias that shifts only the selection) with E4M3 activations,
    in the weights-as-M form and on CTA pairs."""
    w = Workload(f"a8_sigmoid_{rows}", T=rows, D=256, E=16, F=256, k=4, S=256, mode=3,
                 gamma=0.0, dtype="bf16", alpha=0.01, bias="zipf1.1", sel_bias=True,
                 weights="e4m3", acts="e4m3")
    plan = B.launch_plan(B.config_of(w))
    assert plan["w8a8_swap"] == (rows == 200) and plan["pair_routed"] == (rows == 9000)
    _, inp, outs, code = parity.run(w, seed=41)
    assert code == B.MOE_DEVICE_OK
    _check_quantized_rows(w, inp, outs, max_rows=4096)
    rep = parity.check(w, inp, outs, e4m3=True, a8=True, coverage=rows > 4096, y_sample_n=96)
    print(w.name, rep)
