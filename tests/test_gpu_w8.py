"""E4M3 expert weights (moe_quantize_e4m3_rows, moe_forward_w8) against the
CPU oracle, through the C ABI.

The quantizer's codes and scales must equal the oracle's bit for bit.  For
the layer, the library quantizes the seeded bf16 weights itself and the
oracle quantizes the same bf16 weights with its own code; routing is checked
as for bf16 weights and y against the oracle's fp64 layer on the dequantized
weights, at the bf16 tolerance."""
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


@pytest.mark.parametrize("shape", [(300, 192), (4, 64, 128), (3, 2048)])
def test_quantizer_matches_oracle(shape):
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    W = torch.randn(shape, generator=g, device="cuda")
    rows = W.numel() // shape[-1]
    W2 = W.view(rows, shape[-1])
    W2 *= torch.exp(torch.linspace(-12, 6, rows, device="cuda"))[:, None]
    W2[1] = 0.0                      # an all-zero row
    W2[2, :4] = torch.tensor([1e-20, -1e-20, 0.0, -0.0])
    W = W.to(torch.bfloat16)
    q, s = B.quantize_e4m3_rows(W)
    q_ref, s_ref = oracle.quantize_e4m3_rows(W.float().cpu().numpy().reshape(rows, shape[-1]))
    np.testing.assert_array_equal(s.cpu().numpy().reshape(rows), s_ref)
    np.testing.assert_array_equal(q.cpu().numpy().reshape(rows, shape[-1]), q_ref)


# name, T, D, E, F, k, S, mode, gamma, bias
CASES = [
    # shared expert narrower than the routed ones; 16 token tiles for it
    ("w8_multi_tile_top2", 1000, 256, 8, 384, 2, 192, 0, 0.0, "none"),
    # F = 320 and D = 192 leave partial feature tiles; capacity drops
    ("w8_ragged_capacity_e16", 777, 192, 16, 320, 4, 0, 1, 0.75, "normal_var2"),
    # decode-like: 64 experts, shared down projection cut into S / F = 8 pieces
    ("w8_decode_e64_shared_pieces", 64, 512, 64, 128, 8, 1024, 2, 0.0, "zipf1.1"),
    # k = 1 without a shared expert: the down projection writes y
    ("w8_top1_direct_y", 300, 256, 8, 256, 1, 0, 1, 1.0, "normal_var2"),
    # one token, wide d_model (two 256-feature tiles and a ragged one)
    ("w8_one_token_wide", 1, 1088, 8, 192, 2, 320, 0, 0.0, "none"),
    # segments of ~250 rows: several 64-row token tiles per expert
    ("w8_long_segments", 500, 128, 4, 128, 2, 0, 0, 0.0, "none"),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_w8_layers(case):
    name, T, D, E, F, k, S, mode, gamma, bias = case
    w = Workload(name, T=T, D=D, E=E, F=F, k=k, S=S, mode=mode, gamma=gamma, dtype="bf16",
                 alpha=0.01, bias=bias, weights="e4m3")
    _, inp, outs, code = parity.run(w, seed=17)
    assert code == B.MOE_DEVICE_OK
    print(name, parity.check(w, inp, outs, e4m3=True))


def test_w8_zero_tokens():
    w = Workload("w8_empty", T=0, D=128, E=8, F=128, k=2, S=64, mode=0, gamma=1.0,
                 weights="e4m3")
    cfg = B.config_of(w)
    inp = B.quantize_expert_weights(make_inputs(w, 0, "cuda"))
    outs = B.alloc_outputs(cfg)
    outs["expert_counts"].fill_(7)
    outs["aux_loss"].fill_(3.0)
    B.forward(cfg, inp, outs)
    torch.cuda.synchronize()
    assert int(outs["expert_counts"].abs().sum()) == 0
    assert float(outs["aux_loss"][0]) == 0.0


def test_w8_rejects_fp32_layers():
    cfg = B.make_config(16, 64, 4, 64, 2, dtype="fp32")
    with pytest.raises(B.MoeError) as ei:
        B.moe_forward_w8(cfg, *([None] * 23), torch.empty(1 << 20, dtype=torch.uint8,
                                                          device="cuda"))
    assert ei.value.status == B.MOE_ERR_UNSUPPORTED


@pytest.mark.parametrize("name", ["mixtral_decode_fp8", "qwen2_57b_decode_fp8",
                                  "dsv3_decode_fp8"])
def test_w8_benchmark_sized_decode(name):
    w = WORKLOADS[name]
    _, inp, outs, code = parity.run(w)
    assert code == B.MOE_DEVICE_OK
    # decode-sized: scores, routing and y on every token
    rep = parity.check(w, inp, outs, e4m3=True)
    assert rep["y_rows"] == w.T
    print(name, rep)
    del inp, outs
    torch.cuda.empty_cache()
