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
# latent layers: the projection x_lat = x W_in^T is stored in the layer's
# dtype before the router reads it; its bf16 rounding is at most 2^-8 of an
# element (2^-24 in fp32), and the fp32 accumulation adds far less
TOL_X_LAT = {"bf16": 1.1 * 2.0 ** -8, "fp32": 1e-5}
TOL_W = 1e-5
TOL_AUX = 1e-5


def f32(t):
    # copied to the host first, then widened (exact for bf16 and fp32)
    return t.detach().cpu().float().numpy()


def run(w, seed=0, inputs=None, stream=None):
    """Runs the layer; returns (cfg, inputs, outputs, device status).  For
    E4M3 workloads the library quantizes the bf16 weights first and the
    returned inputs are the bf16 ones (the oracle quantizes them itself)."""
    cfg = B.config_of(w)
    inp = inputs if inputs is not None else make_inputs(w, seed, "cuda")
    run_inp = (B.quantize_expert_weights(inp, stream, a8=w.acts == "e4m3")
               if w.weights == "e4m3" else inp)
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


BLOCK = 128


def coverage_sample(w, idx, dropped, n_min=512, seed=0):
    """A seeded token sample whose y rows touch every tile any launch can
    cut the layer into.

    The expert-contiguous layout keeps each expert's kept assignments in
    token order, so assignment (t, j) to expert e sits at position p = the
    number of earlier tokens kept by e.  Every tile of the grouped GEMMs
    (128-row tiles, 256-row pair tiles, a segment's leftover rows) is a union
    of 128-position blocks of one segment, starting at a multiple of 128.
    The sample holds:
      - the first and last kept token of every expert;
      - for every 128-position block of every segment, at least one token
        (a random one of the block, unless an earlier pick already lands in
        it; each token covers the blocks of all its k assignments);
      - a token of every 128-token block of the batch (the shared expert's
        dense tiles);
      - up to 8 tokens that lost an expert to capacity;
      - random tokens up to n_min.
    Returns the sorted token indices."""
    rng = np.random.default_rng(seed)
    T, k = idx.shape
    if T == 0:
        return np.zeros(0, dtype=np.int64)
    t_all = np.repeat(np.arange(T), k)
    e_all = idx.ravel().astype(np.int64)
    kept = dropped.ravel() == 0
    t_k, e_k = t_all[kept], e_all[kept]
    order = np.lexsort((t_k, e_k))            # by expert, then token
    t_s, e_s = t_k[order], e_k[order]
    start = np.searchsorted(e_s, np.arange(w.E))
    end = np.searchsorted(e_s, np.arange(w.E), side="right")
    pos = np.arange(t_s.size) - start[e_s]
    blk = e_s * (T // BLOCK + 2) + pos // BLOCK   # (expert, block) key
    # the (expert, block) keys each token covers
    key_of_tok = {}
    for t, key in zip(t_s.tolist(), blk.tolist()):
        key_of_tok.setdefault(t, []).append(key)
    covered, pick = set(), set()

    def take(t):
        if t not in pick:
            pick.add(t)
            covered.update(key_of_tok.get(t, ()))

    for e in range(w.E):
        if end[e] > start[e]:
            take(int(t_s[start[e]]))
            take(int(t_s[end[e] - 1]))
    ukeys, first = np.unique(blk, return_index=True)
    counts = np.diff(np.append(first, blk.size))
    for key, f, c in zip(ukeys.tolist(), first.tolist(), counts.tolist()):
        if key not in covered:
            take(int(t_s[f + rng.integers(c)]))
    for b0 in range(0, T, BLOCK):
        if not any(b0 <= t < b0 + BLOCK for t in pick):
            take(int(b0 + rng.integers(min(BLOCK, T - b0))))
    drows = np.nonzero(dropped.any(1))[0]
    if drows.size:
        for t in rng.choice(drows, size=min(8, drows.size), replace=False).tolist():
            take(int(t))
    rest = np.setdiff1d(np.arange(T), np.fromiter(pick, dtype=np.int64))
    if len(pick) < n_min and rest.size:
        for t in rng.choice(rest, size=min(n_min - len(pick), rest.size), replace=False):
            take(int(t))
    return np.array(sorted(pick), dtype=np.int64)


def e4m3_weights(W):
    """The oracle's own E4M3 codes and scales of a bf16 weight matrix (device
    tensor [rows, cols]): (codes, scales) as numpy arrays."""
    return oracle.quantize_e4m3_rows(f32(W))


def check(w, inp, outs, sample=None, logit_rows=None, y_sample_n=None, seed=0, e4m3=False,
          coverage=False, a8=False):
    """Asserts every parity criterion; returns a dict of the measured errors.
    coverage: y on coverage_sample's tokens (at least y_sample_n, default
    512) instead of a plain random sample.
    e4m3: the layer ran with E4M3 expert weights; the oracle quantizes the
    same bf16 weights itself and computes with the dequantized values.
    a8: E4M3 activations too (the oracle's swiglu_rows_w8a8)."""
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

    # 1. router scores against the oracle's own.  A latent layer's router
    # reads the stored x_lat = x W_in^T; the oracle's router takes the GPU's
    # own x_lat rows (widened exactly), and x_lat is checked against the
    # oracle's projection separately, at the bound of its storage rounding.
    rows = np.arange(T) if logit_rows is None else np.asarray(logit_rows)
    if rows.size:
        sel_rows = torch.as_tensor(rows, device=inp["x"].device)
        if latent:
            x_lat, _ = B.latent_activations(B.config_of(w), w.D_outer, outs["workspace"])
            xr = f32(x_lat[sel_rows]).astype(np.float64)
            lat_ref = layer_input(f32(inp["x"][sel_rows]))
            rep["x_lat_rel"] = float(np.abs(xr - lat_ref).max() /
                                     max(np.abs(lat_ref).max(), 1e-30))
            assert rep["x_lat_rel"] <= TOL_X_LAT[w.dtype], rep
        else:
            xr = f32(inp["x"][sel_rows])
        s_ref = oracle.linear(xr, f32(inp["W_r"]))
        if b is not None and not w.sel_bias:
            s_ref = s_ref + b.astype(np.float64)
        den = max(np.abs(s_ref).max(), 1e-30)
        rep["logits_rel"] = float(np.abs(s_gpu[rows] - s_ref).max() / den)
        assert rep["logits_rel"] <= TOL_LOGITS, rep

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
    if sample is None and coverage:
        sample = coverage_sample(w, idx, dropped, n_min=y_sample_n or 512, seed=seed)
    elif sample is None:
        sample = (np.arange(T) if y_sample_n is None
                  else pick_sample(w, dropped, idx, None, y_sample_n, seed))
    sel = torch.as_tensor(sample, device=inp["x"].device)
    x_rows = layer_input(f32(inp["x"][sel]))
    Wg, Wu, Wd = inp["W_gate"], inp["W_up"], inp["W_down"]
    if e4m3:
        def weights(*Ws):
            return tuple(a for W in Ws for a in e4m3_weights(W)) + (("a8",) if a8 else ())
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
