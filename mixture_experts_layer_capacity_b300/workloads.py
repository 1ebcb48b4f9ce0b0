"""Synthetic workloads and their seeded input generators.

This module holds shapes, seeds and random draws only -- none of the layer's
arithmetic.  The CUDA path and the tests (which hand the same tensors to the
CPU oracle) both take their inputs from here.

Recipe: one ``torch.Generator`` per tensor on the target device, seeded
``seed * 100 + tensor_id`` with ids x=0, W_r=1, b_r=2, W_gate=3, W_up=4,
W_down=5, Ws_gate=6, Ws_up=7, Ws_down=8, W_in=9, W_out=10.  Each draw is fp32 N(0, 1), scaled by
the standard deviation and cast to the workload dtype.  Stacked expert weights
are drawn one expert at a time from that tensor's generator (so the fp32
temporary stays one expert large).  x ~ N(0, 1); every weight ~ N(0, 1/d_in)
where d_in is the reduction dimension (D for W_r, W_gate, W_up, Ws_gate,
Ws_up; F for W_down; S for Ws_down; D_outer for W_in; D for W_out).

A latent workload (D_outer > 0) runs the layer at width D on x W_in^T, with
x [T, D_outer], W_in [D, D_outer] and W_out [D_outer, D].

Weight layout (reduction dimension contiguous, "K-major"):
  W_r [E, D]; W_gate, W_up [E, F, D]; W_down [E, D, F];
  Ws_gate, Ws_up [S, D]; Ws_down [D, S].
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch

GATING_SOFTMAX_SELECTED = 0      # Mixtral: softmax over the k chosen scores
GATING_SOFTMAX_ALL = 1           # Switch / Qwen2: softmax over all, keep k
GATING_SOFTMAX_ALL_RENORM = 2    # softmax over all, renormalised over the k
GATING_SIGMOID_SELECTED = 3      # sigmoid of each score, normalised over the k


@dataclass(frozen=True)
class Workload:
    name: str
    T: int            # tokens
    D: int            # d_model
    E: int            # routed experts
    F: int            # d_expert (hidden width of one routed expert)
    k: int            # experts per token
    S: int = 0        # hidden width of the shared expert; 0 = none
    mode: int = GATING_SOFTMAX_SELECTED
    gamma: float = 0.0    # capacity factor; <= 0 = dropless
    dtype: str = "bf16"   # "bf16" or "fp32"
    alpha: float = 0.01   # balance-loss coefficient
    bias: str = "none"    # router logit bias: "none", "normal_var2", "zipf1.1"
    sel_bias: bool = False  # the bias shifts only the top-k selection keys
    D_outer: int = 0      # latent MoE: outer width (x and y); 0 = plain layer
    weights: str = "bf16"  # expert weight storage: "bf16", or "e4m3" (row-scaled FP8,
                           # quantized from the same seeded bf16 weights)
    acts: str = "bf16"     # expert GEMM activations: "bf16", or "e4m3" (row-scaled FP8
                           # token and hidden rows; needs weights="e4m3")
    description: str = ""

    def with_T(self, T: int) -> "Workload":
        return replace(self, T=T, name=f"{self.name.split('@')[0]}@T={T}")

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32


WORKLOADS = {
    "tiny_fp32": Workload(
        "tiny_fp32", T=256, D=64, E=4, F=128, k=2, S=0,
        mode=GATING_SOFTMAX_SELECTED, gamma=0.0, dtype="fp32",
        description="tiny fp32 layer, top-2 softmax over selected, dropless"),
    "switch_top1_capacity": Workload(
        "switch_top1_capacity", T=4096, D=512, E=8, F=2048, k=1, S=0,
        mode=GATING_SOFTMAX_ALL, gamma=1.0, dtype="bf16", alpha=0.01,
        bias="normal_var2",
        description="Switch-style top-1, raw probability, capacity factor 1.0 "
                    "with token-order drops, biased router for imbalance"),
    "mixtral_prefill": Workload(
        "mixtral_prefill", T=8192, D=4096, E=8, F=14336, k=2,
        mode=GATING_SOFTMAX_SELECTED, description="Mixtral-8x7B-shaped, T=8192"),
    "mixtral_decode": Workload(
        "mixtral_decode", T=64, D=4096, E=8, F=14336, k=2,
        mode=GATING_SOFTMAX_SELECTED, description="Mixtral-8x7B-shaped, T=64"),
    "qwen2_57b_prefill": Workload(
        "qwen2_57b_prefill", T=8192, D=3584, E=64, F=2560, k=8, S=20480,
        mode=GATING_SOFTMAX_ALL,
        description="Qwen2-57B-A14B-shaped, shared expert d=20480, T=8192"),
    "qwen2_57b_decode": Workload(
        "qwen2_57b_decode", T=64, D=3584, E=64, F=2560, k=8, S=20480,
        mode=GATING_SOFTMAX_ALL,
        description="Qwen2-57B-A14B-shaped, shared expert d=20480, T=64"),
    "dsv3_prefill": Workload(
        "dsv3_prefill", T=16384, D=7168, E=256, F=2048, k=8, S=2048,
        mode=GATING_SOFTMAX_ALL_RENORM, bias="zipf1.1",
        description="DeepSeek-V3-shaped, renormalised top-8, Zipf-skewed bias, T=16384"),
    # the DeepSeek-V3 widths with 32 experts and T=4096 (2.9 GB of weights):
    # a profiling case for the CTA-pair GEMMs (256-row tiles and swap units)
    # small enough for multi-pass counter captures
    "dsv3_prefill_e32": Workload(
        "dsv3_prefill_e32", T=4096, D=7168, E=32, F=2048, k=8, S=2048,
        mode=GATING_SOFTMAX_ALL_RENORM, bias="zipf1.1",
        description="DeepSeek-V3 widths, 32 experts, T=4096: profiling case"),
    # the same profiling case with E4M3 weights and activations
    "dsv3_prefill_e32_w8a8": Workload(
        "dsv3_prefill_e32_w8a8", T=4096, D=7168, E=32, F=2048, k=8, S=2048,
        mode=GATING_SOFTMAX_ALL_RENORM, bias="zipf1.1", weights="e4m3", acts="e4m3",
        description="DeepSeek-V3 widths, 32 experts, T=4096, E4M3 weights and "
                    "activations: profiling case"),
    "dsv3_decode": Workload(
        "dsv3_decode", T=64, D=7168, E=256, F=2048, k=8, S=2048,
        mode=GATING_SOFTMAX_ALL_RENORM, bias="zipf1.1",
        description="DeepSeek-V3-shaped, renormalised top-8, Zipf-skewed bias, T=64"),
    # latent MoE with the page's widths (4096 down to 1024 and back); the
    # expert count, width and k are this build's choice (not on the pages)
    "latent_prefill": Workload(
        "latent_prefill", T=4096, D=1024, E=64, F=2048, k=8, D_outer=4096,
        mode=GATING_SOFTMAX_ALL_RENORM,
        description="latent MoE: 4096 -> 1024, 64 experts d=2048, top-8, -> 4096, T=4096"),
    "latent_decode": Workload(
        "latent_decode", T=64, D=1024, E=64, F=2048, k=8, D_outer=4096,
        mode=GATING_SOFTMAX_ALL_RENORM,
        description="latent MoE: 4096 -> 1024, 64 experts d=2048, top-8, -> 4096, T=64"),
    # the decode shapes with E4M3 expert weights (one fp32 scale per weight row)
    "mixtral_decode_fp8": Workload(
        "mixtral_decode_fp8", T=64, D=4096, E=8, F=14336, k=2,
        mode=GATING_SOFTMAX_SELECTED, weights="e4m3",
        description="Mixtral-8x7B-shaped, T=64, E4M3 expert weights"),
    "qwen2_57b_decode_fp8": Workload(
        "qwen2_57b_decode_fp8", T=64, D=3584, E=64, F=2560, k=8, S=20480,
        mode=GATING_SOFTMAX_ALL, weights="e4m3",
        description="Qwen2-57B-A14B-shaped, T=64, E4M3 expert weights"),
    "dsv3_decode_fp8": Workload(
        "dsv3_decode_fp8", T=64, D=7168, E=256, F=2048, k=8, S=2048,
        mode=GATING_SOFTMAX_ALL_RENORM, bias="zipf1.1", weights="e4m3",
        description="DeepSeek-V3-shaped, T=64, E4M3 expert weights"),
    # E4M3 token and hidden rows as well as E4M3 expert weights (both GEMM
    # operands in FP8 on the tensor cores)
    "mixtral_decode_w8a8": Workload(
        "mixtral_decode_w8a8", T=64, D=4096, E=8, F=14336, k=2,
        mode=GATING_SOFTMAX_SELECTED, weights="e4m3", acts="e4m3",
        description="Mixtral-8x7B-shaped, T=64, E4M3 expert weights and activations"),
    "qwen2_57b_decode_w8a8": Workload(
        "qwen2_57b_decode_w8a8", T=64, D=3584, E=64, F=2560, k=8, S=20480,
        mode=GATING_SOFTMAX_ALL, weights="e4m3", acts="e4m3",
        description="Qwen2-57B-A14B-shaped, T=64, E4M3 expert weights and activations"),
    "dsv3_decode_w8a8": Workload(
        "dsv3_decode_w8a8", T=64, D=7168, E=256, F=2048, k=8, S=2048,
        mode=GATING_SOFTMAX_ALL_RENORM, bias="zipf1.1", weights="e4m3", acts="e4m3",
        description="DeepSeek-V3-shaped, T=64, E4M3 expert weights and activations"),
    "dsv3_prefill_w8a8": Workload(
        "dsv3_prefill_w8a8", T=16384, D=7168, E=256, F=2048, k=8, S=2048,
        mode=GATING_SOFTMAX_ALL_RENORM, bias="zipf1.1", weights="e4m3", acts="e4m3",
        description="DeepSeek-V3-shaped, T=16384, E4M3 expert weights and activations"),
    "dsv3_sigmoid_decode": Workload(
        "dsv3_sigmoid_decode", T=64, D=7168, E=256, F=2048, k=8, S=2048,
        mode=GATING_SIGMOID_SELECTED, bias="zipf1.1", sel_bias=True,
        description="DeepSeek-V3-shaped with its own gating: sigmoid scores "
                    "normalised over the chosen 8, Zipf-skewed selection-only bias, T=64"),
}

_TID = {"x": 0, "W_r": 1, "b_r": 2, "W_gate": 3, "W_up": 4, "W_down": 5,
        "Ws_gate": 6, "Ws_up": 7, "Ws_down": 8, "W_in": 9, "W_out": 10}


def _gen(device, seed, name):
    g = torch.Generator(device=device)
    g.manual_seed(seed * 100 + _TID[name])
    return g


def _normal(shape, std, g, device, dtype):
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32)
            * std).to(dtype)


def _stacked(E, rows, cols, std, g, device, dtype):
    out = torch.empty((E, rows, cols), device=device, dtype=dtype)
    for e in range(E):
        out[e] = _normal((rows, cols), std, g, device, dtype)
    return out


def make_inputs(w: Workload, seed: int = 0, device="cuda", weights: bool = True):
    """Seeded synthetic inputs for workload ``w`` on ``device``.

    Returns a dict with x, W_r, b_r (None if the workload has no bias), and,
    when ``weights`` is true, W_gate, W_up, W_down, Ws_gate, Ws_up, Ws_down
    (the shared ones None when S = 0).  b_r is fp32; the rest use the
    workload dtype.
    """
    dt = w.torch_dtype
    dev = torch.device(device)
    out = {}
    out["x"] = _normal((w.T, w.D_outer or w.D), 1.0, _gen(dev, seed, "x"), dev, dt)
    if w.D_outer:
        out["W_in"] = _normal((w.D, w.D_outer), 1.0 / math.sqrt(w.D_outer),
                              _gen(dev, seed, "W_in"), dev, dt)
        out["W_out"] = _normal((w.D_outer, w.D), 1.0 / math.sqrt(w.D),
                               _gen(dev, seed, "W_out"), dev, dt)
    out["W_r"] = _normal((w.E, w.D), 1.0 / math.sqrt(w.D), _gen(dev, seed, "W_r"), dev, dt)
    if w.bias == "normal_var2":
        out["b_r"] = _normal((w.E,), math.sqrt(2.0), _gen(dev, seed, "b_r"), dev,
                             torch.float32)
    elif w.bias == "zipf1.1":
        # log of a Zipf(1.1) weight per expert: low-numbered experts favoured.
        out["b_r"] = (-1.1 * torch.log(torch.arange(1, w.E + 1, dtype=torch.float64))
                      ).to(torch.float32).to(dev)
    else:
        out["b_r"] = None
    if not weights:
        return out
    sD, sF = 1.0 / math.sqrt(w.D), 1.0 / math.sqrt(w.F)
    out["W_gate"] = _stacked(w.E, w.F, w.D, sD, _gen(dev, seed, "W_gate"), dev, dt)
    out["W_up"] = _stacked(w.E, w.F, w.D, sD, _gen(dev, seed, "W_up"), dev, dt)
    out["W_down"] = _stacked(w.E, w.D, w.F, sF, _gen(dev, seed, "W_down"), dev, dt)
    if w.S > 0:
        sS = 1.0 / math.sqrt(w.S)
        out["Ws_gate"] = _normal((w.S, w.D), sD, _gen(dev, seed, "Ws_gate"), dev, dt)
        out["Ws_up"] = _normal((w.S, w.D), sD, _gen(dev, seed, "Ws_up"), dev, dt)
        out["Ws_down"] = _normal((w.D, w.S), sS, _gen(dev, seed, "Ws_down"), dev, dt)
    else:
        out["Ws_gate"] = out["Ws_up"] = out["Ws_down"] = None
    return out
