"""Parity checks of the CUDA path (called through the C ABI) against the CPU
oracle on the same seeded inputs.

Criteria:
  - router scores: max|s_gpu - s_oracle| / max|s_oracle| <= 1e-3;
  - routing is re-derived by the oracle from the GPU's own scores (so that
    near-ties are judged on identical values), then topk_idx, dropped_mask,
    expert_counts and kept_counts must match bit for bit;
  - topk_w within 1e-5 absolute; aux_loss within 1e-5 relative;
  - y: max|y_gpu - y_oracle| / max|y_oracle| <= 2e-2 (bf16), 1e-4 (fp32),
    on every token for small layers and on a seeded sample for large ones
    (y is per token once routing is fixed, so sampled rows are exact checks).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from mixture_experts_layer_capacity_b300 import binding as B
from mixture_experts_layer_capacity_b300.workloads import make_inputs

TOL_Y = {"bf16": 2e-2, "fp32": 1e-4}
TOL_LOGITS = 1e-3
# latent bf16 layers: the router reads x W_in^T rounded to bf16 (unit roundoff
# 2^-8 per element), which the fp64 oracle does not round; the scores' error
# relative to their maximum stays within a few of those units
TOL_LOGITS_LATENT_BF16 = 1e-2
TOL_W = 1e-5
TOL_AUX = 1e-5


def f32(t):
    return t.detach().float().cpu().numpy()


def run(w, seed=0, inputs=None, stream=None):
    """Runs the layer; returns (cfg, inputs, outputs, device status).  For
    E4M3 workloads the library quantizes the bf16 weights first and the
    returned inputs are the bf16 ones (the oracle quantizes them itself)."""
    cfg = B.config_of(w)
    inp = inputs if inputs is not None else make_inputs(w, seed, "cuda")
    run_inp = B.quantize_expert_weights(inp, stream) if w.weights == "e4m3" else inp
    outs = B.forward(cfg, run_inp, stream=stream)
    code = B.read_device_status(cfg, outs["workspace"], stream=stream)
    return cfg, inp, outs, code


def pick_sample(w, dropped, idx, kept_mask_rows, n, seed=0):
    """Seeded token sample; with capacity it includes the busiest expert's
    first and last kept token and some tokens that lost an expert."""
    rng = np.random.default_rng(seed)
    T = w.T
    pick = set(rng.choice(T, size=min(n, T), replace=False).tolist())
    if w.gamma > 0 and T > 0:
        counts = np.bincount(idx.ravel(), minlength=w.E)
        busiest = int(np.argmax(counts))
        rows, slots = np.nonzero((idx == busiest) & (dropped == 0))
        if rows.size:
            pick |= {int(rows.min()), int(rows.max())}
        drows = np.nonzero(dropped.any(1))[0]
        if drows.size:
            pick |= set(rng.choice(drows, size=min(4, drows.size), replace=False).tolist())
    return np.array(sorted(pick), dtype=np.int64)


def e4m3_weights(W):
    """The oracle's own E4M3 codes and scales of a bf16 weight matrix (device
    tensor [rows, cols]): (codes, scales) as numpy arrays."""
    return oracle.quantize_e4m3_rows(f32(W))


def check(w, inp, outs, sample=None, logit_rows=None, y_sample_n=None, seed=0, e4m3=False):
    """Asserts every parity criterion; returns a dict of the measured errors.
    e4m3: the layer ran with E4M3 expert weights; the oracle quantizes the
    same bf16 weights itself and computes with the dequantized values."""
    T, E, k = w.T, w.E, w.k
    gamma32 = float(np.float32(w.gamma))
    alpha32 = float(np.float32(w.alpha))
    s_gpu = outs["router_logits"].cpu().double().numpy()
    b = None if inp.get("b_r") is None else f32(inp["b_r"])
    rep = {}

    latent = inp.get("W_in") is not None

    def layer_input(rows_x):
        """The layer's input rows: x, or x W_in^T (fp64) for a latent layer."""
        return oracle.linear(rows_x, f32(inp["W_in"])) if latent else rows_x

    # 1. router scores against the oracle's own
    rows = np.arange(T) if logit_rows is None else np.asarray(logit_rows)
    if rows.size:
        xr = layer_input(f32(inp["x"][torch.as_tensor(rows, device=inp["x"].device)]))
        s_ref = oracle.linear(xr, f32(inp["W_r"]))
        if b is not None and not w.sel_bias:
            s_ref = s_ref + b.astype(np.float64)
        den = max(np.abs(s_ref).max(), 1e-30)
        rep["logits_rel"] = float(np.abs(s_gpu[rows] - s_ref).max() / den)
        tol = TOL_LOGITS_LATENT_BF16 if latent and w.dtype == "bf16" else TOL_LOGITS
        assert rep["logits_rel"] <= tol, rep

    # 2. routing, capacity and statistics re-derived from the GPU scores
    idx, wts, P_sum, counts = oracle.route(s_gpu, k, w.mode,
                                           sel_bias=b if w.sel_bias else None)
    C = oracle.capacity(T, k, E, gamma32)
    dropped, kept = oracle.apply_capacity(idx, E, C)
    aux = oracle.aux_loss(T, k, E, alpha32, counts, P_sum)
    np.testing.assert_array_equal(outs["topk_idx"].cpu().numpy(), idx)
    np.testing.assert_array_equal(outs["dropped_mask"].cpu().numpy(), dropped)
    np.testing.assert_array_equal(outs["expert_counts"].cpu().numpy(), counts)
    np.testing.assert_array_equal(outs["kept_counts"].cpu().numpy(), kept)
    if T:
        rep["w_abs"] = float(np.abs(outs["topk_w"].cpu().double().numpy() - wts).max())
        assert rep["w_abs"] <= TOL_W, rep
    aux_gpu = float(outs["aux_loss"].cpu()[0])
    rep["aux_rel"] = abs(aux_gpu - aux) / max(abs(aux), 1e-12)
    assert abs(aux_gpu - aux) <= TOL_AUX * abs(aux) + 1e-9, (aux_gpu, aux)

    # 3. y on all tokens or a sample
    if T == 0:
        return rep
    if sample is None:
        sample = (np.arange(T) if y_sample_n is None
                  else pick_sample(w, dropped, idx, None, y_sample_n, seed))
    sel = torch.as_tensor(sample, device=inp["x"].device)
    x_rows = layer_input(f32(inp["x"][sel]))
    Wg, Wu, Wd = inp["W_gate"], inp["W_up"], inp["W_down"]
    if e4m3:
        def weights(*Ws):
            return tuple(a for W in Ws for a in e4m3_weights(W))
    else:
        def weights(*Ws):
            return tuple(f32(W) for W in Ws)
    shared = None
    if w.S > 0:
        shared = weights(inp["Ws_gate"], inp["Ws_up"], inp["Ws_down"])
    y_ref = oracle.moe_rows(x_rows, idx[sample], wts[sample], dropped[sample],
                            lambda e: weights(Wg[e], Wu[e], Wd[e]), shared=shared)
    if latent:
        y_ref = oracle.linear(y_ref, f32(inp["W_out"]))
    y_gpu = f32(outs["y"][sel]).astype(np.float64)
    den = max(np.abs(y_ref).max(), 1e-30)
    rep["y_rel"] = float(np.abs(y_gpu - y_ref).max() / den)
    rep["y_rows"] = int(len(sample))
    assert rep["y_rel"] <= TOL_Y[w.dtype], rep
    return rep
