"""Pins of the CPU oracle to what the pages and the mathematics fix.

Each test ties the oracle to something other than itself: a worked example
printed on the pages, a closed form, an exercise, an independent brute force
(numpy matrix products, a full sort, an explicit recount), or an invariant.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle

from conftest import GOLDEN


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _silu(a):
    return a / (1.0 + np.exp(-a))


def _dense_swiglu(X, Wg, Wu, Wd):
    """numpy matrix form of one SwiGLU network over all rows of X (fp64)."""
    X = X.astype(np.float64)
    return (_silu(X @ Wg.astype(np.float64).T) * (X @ Wu.astype(np.float64).T)) \
        @ Wd.astype(np.float64).T


def _rand_layer(rng, T, D, E, F, S=0):
    x = rng.standard_normal((T, D)).astype(np.float32)
    Wr = (rng.standard_normal((E, D)) / math.sqrt(D)).astype(np.float32)
    Wg = (rng.standard_normal((E, F, D)) / math.sqrt(D)).astype(np.float32)
    Wu = (rng.standard_normal((E, F, D)) / math.sqrt(D)).astype(np.float32)
    Wd = (rng.standard_normal((E, D, F)) / math.sqrt(F)).astype(np.float32)
    sh = {}
    if S:
        sh = dict(Ws_gate=(rng.standard_normal((S, D)) / math.sqrt(D)).astype(np.float32),
                  Ws_up=(rng.standard_normal((S, D)) / math.sqrt(D)).astype(np.float32),
                  Ws_down=(rng.standard_normal((D, S)) / math.sqrt(S)).astype(np.float32))
    return x, Wr, Wg, Wu, Wd, sh


# --- gating -----------------------------------------------------------------

@pytest.mark.parametrize("mode", [0, 1, 2])
def test_worked_example(mode):
    g = _load("worked_example.json")
    p = np.array(g["probs"])
    s = np.log(p)[None, :]
    idx, w, P_sum, counts = oracle.route(s, g["k"], mode)
    assert idx[0].tolist() == g["chosen"]
    if mode in (0, 2):
        np.testing.assert_allclose(w[0], g["weights_renormalised"], rtol=0, atol=1e-12)
    else:
        # softmax over all, no renormalisation: the raw probabilities, sum < 1
        np.testing.assert_allclose(w[0], p[g["chosen"]], rtol=0, atol=1e-12)
        assert abs(w[0].sum() - g["selected_prob_sum"]) < 1e-12
    np.testing.assert_allclose(P_sum, p, atol=1e-12)


def test_selected_softmax_sums_to_one_and_modes_agree():
    rng = np.random.default_rng(1)
    s = rng.standard_normal((500, 16)) * 3
    for k in (1, 2, 5, 16):
        _, w0, _, _ = oracle.route(s, k, 0)
        _, w1, _, _ = oracle.route(s, k, 1)
        _, w2, _, _ = oracle.route(s, k, 2)
        np.testing.assert_allclose(w0.sum(1), 1.0, atol=1e-12)
        np.testing.assert_allclose(w2.sum(1), 1.0, atol=1e-12)
        # modes 0 and 2 are the same function in exact arithmetic
        np.testing.assert_allclose(w0, w2, atol=1e-12)
        assert np.all(w1.sum(1) <= 1.0 + 1e-12)
        if k == 16:
            np.testing.assert_allclose(w1.sum(1), 1.0, atol=1e-12)


def test_mode1_weights_are_softmax_probabilities():
    rng = np.random.default_rng(2)
    s = rng.standard_normal((64, 12)) * 2
    idx, w, P_sum, _ = oracle.route(s, 3, 1)
    z = np.exp(s - s.max(1, keepdims=True))
    p = z / z.sum(1, keepdims=True)
    np.testing.assert_allclose(w, np.take_along_axis(p, idx.astype(np.int64), 1), atol=1e-14)
    np.testing.assert_allclose(P_sum, p.sum(0), atol=1e-12)


def test_top1_renormalised_weight_is_exactly_one():
    rng = np.random.default_rng(3)
    s = rng.standard_normal((100, 8))
    _, w, _, _ = oracle.route(s, 1, 2)
    assert np.all(w == 1.0)
    _, w1, _, _ = oracle.route(s, 1, 1)
    z = np.exp(s - s.max(1, keepdims=True))
    np.testing.assert_allclose(w1[:, 0], (z / z.sum(1, keepdims=True)).max(1), atol=1e-14)


@pytest.mark.parametrize("E,k", [(5, 1), (5, 2), (6, 3), (8, 8), (16, 4)])
def test_topk_against_full_sort_with_ties(E, k):
    rng = np.random.default_rng(E * 10 + k)
    # small integers: many exact ties, the order must go to the lower index
    s = rng.integers(-2, 3, size=(300, E)).astype(np.float64)
    idx, _, _, counts = oracle.route(s, k, 1)
    for t in range(s.shape[0]):
        want = sorted(range(E), key=lambda e: (-s[t, e], e))[:k]
        assert idx[t].tolist() == want
    assert counts.sum() == s.shape[0] * k
    np.testing.assert_array_equal(counts, np.bincount(idx.ravel(), minlength=E))


def test_topk_maximises_subset_sum():
    rng = np.random.default_rng(7)
    E = 6
    s = rng.standard_normal((50, E))
    for k in (1, 2, 3, 4):
        idx, _, _, _ = oracle.route(s, k, 0)
        for t in range(s.shape[0]):
            best = max(sum(s[t, list(c)]) for c in itertools.combinations(range(E), k))
            assert abs(sum(s[t, idx[t]]) - best) < 1e-12
            assert len(set(idx[t].tolist())) == k


def test_nonfinite_scores_rejected():
    s = np.zeros((2, 4))
    s[1, 2] = np.nan
    with pytest.raises(RuntimeError):
        oracle.route(s, 2, 0)


# --- balance loss -----------------------------------------------------------

def test_balance_loss_closed_forms():
    g = _load("balance_loss_exercise.json")
    E, k, alpha = g["E"], g["k"], g["alpha"]
    T = 8 * E
    # even split: token t strongly prefers expert t % E (probability ~ 1)
    s = np.zeros((T, E))
    s[np.arange(T), np.arange(T) % E] = 60.0
    idx, _, P_sum, counts = oracle.route(s, k, 1)
    assert np.all(counts == T // E)
    assert abs(oracle.aux_loss(T, k, E, alpha, counts, P_sum) - g["even_split"]) < 1e-12
    # collapse: every token to expert 0 with probability 1
    s = np.zeros((T, E))
    s[:, 0] = 60.0
    idx, _, P_sum, counts = oracle.route(s, k, 1)
    assert counts[0] == T
    assert abs(oracle.aux_loss(T, k, E, alpha, counts, P_sum)
               - g["all_to_one_expert_prob_one"]) < 1e-12


def test_balance_loss_even_split_top2_is_alpha():
    # f_e counts assignments over T*k, so an even top-2 split still gives alpha
    E, k, T, alpha = 8, 2, 64, 0.01
    s = np.zeros((T, E))
    s[np.arange(T), (2 * np.arange(T)) % E] = 60.0
    s[np.arange(T), (2 * np.arange(T) + 1) % E] = 59.0
    idx, _, P_sum, counts = oracle.route(s, k, 0)
    assert np.all(counts == T * k // E)
    # P_e: each token splits ~ (1, e^-1)/(1+e^-1) between its two experts
    a = oracle.aux_loss(T, k, E, alpha, counts, P_sum)
    assert abs(a - alpha) < 1e-12


def test_balance_loss_zero_tokens():
    assert oracle.aux_loss(0, 2, 4, 0.01, np.zeros(4, np.int64), np.zeros(4)) == 0.0


# --- capacity ---------------------------------------------------------------

def test_capacity_exercise_and_switch_workload():
    g = _load("capacity_exercise.json")
    assert oracle.capacity(g["T"], g["k"], g["E"], g["gamma"]) == g["C"]
    # Switch-style workload: T=4096, top-1, E=8, factor 1.0 -> the fair share
    assert oracle.capacity(4096, 1, 8, 1.0) == 512
    assert oracle.capacity(4096, 1, 8, 0.0) == -1
    assert oracle.capacity(4096, 1, 8, -1.0) == -1
    # rounding up
    assert oracle.capacity(10, 1, 3, 1.0) == 4
    assert oracle.capacity(1, 1, 8, 1.0) == 1


@pytest.mark.parametrize("gamma", [0.25, 0.5, 1.0, 1.25])
def test_capacity_token_order_against_recount(gamma):
    rng = np.random.default_rng(int(gamma * 100))
    T, E, k = 257, 8, 2
    # skewed scores so that low experts overflow
    s = rng.standard_normal((T, E)) + np.linspace(2, 0, E)
    idx, _, _, counts = oracle.route(s, k, 0)
    C = oracle.capacity(T, k, E, gamma)
    dropped, kept = oracle.apply_capacity(idx, E, C)
    assert np.all(kept <= C)
    assert kept.sum() + dropped.sum() == T * k
    np.testing.assert_array_equal(kept, np.minimum(counts, C))
    # independent recount: the first C tokens (in token order) of each expert stay
    want = np.zeros((T, k), np.uint8)
    for e in range(E):
        rows, slots = np.nonzero(idx == e)
        order = np.argsort(rows, kind="stable")
        rows, slots = rows[order], slots[order]
        want[rows[C:], slots[C:]] = 1
    np.testing.assert_array_equal(dropped, want)


def test_capacity_large_factor_is_dropless():
    rng = np.random.default_rng(5)
    s = rng.standard_normal((100, 4))
    idx, _, _, counts = oracle.route(s, 2, 0)
    d_big, k_big = oracle.apply_capacity(idx, 4, oracle.capacity(100, 2, 4, 1e6))
    d_none, k_none = oracle.apply_capacity(idx, 4, -1)
    assert d_big.sum() == 0 and d_none.sum() == 0
    np.testing.assert_array_equal(k_big, counts)
    np.testing.assert_array_equal(k_none, counts)


# --- experts and the whole layer -----------------------------------------------

def test_router_logits_against_matmul():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((33, 40)).astype(np.float32)
    Wr = rng.standard_normal((7, 40)).astype(np.float32)
    b = rng.standard_normal(7).astype(np.float32)
    s = oracle.router_logits(x, Wr, b)
    np.testing.assert_allclose(s, x.astype(np.float64) @ Wr.astype(np.float64).T + b,
                               rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_single_expert_is_the_dense_mlp(mode):
    rng = np.random.default_rng(20 + mode)
    x, Wr, Wg, Wu, Wd, _ = _rand_layer(rng, 40, 16, 1, 24)
    out = oracle.moe_forward(x, Wr, Wg, Wu, Wd, k=1, mode=mode)
    ref = _dense_swiglu(x, Wg[0], Wu[0], Wd[0])
    np.testing.assert_allclose(out["y"], ref, rtol=1e-11, atol=1e-11)
    assert np.all(out["w"] == 1.0)


def _numpy_layer(x, Wr, Wg, Wu, Wd, k, mode, gamma, sh, sel_bias=None):
    """Brute force: run every expert on every token, then mask by routing.
    sel_bias: a bias that only the ranking sees (key = fp32(s) + fp32(b) in
    fp32)."""
    T, E = x.shape[0], Wr.shape[0]
    s = x.astype(np.float64) @ Wr.astype(np.float64).T
    if mode == 3:
        a = 1.0 / (1.0 + np.exp(-s))
        p = a / a.sum(1, keepdims=True)
    else:
        z = np.exp(s - s.max(1, keepdims=True))
        p = z / z.sum(1, keepdims=True)
    key = s if sel_bias is None else \
        (s.astype(np.float32) + np.asarray(sel_bias, np.float32)).astype(np.float64)
    order = np.array([sorted(range(E), key=lambda e: (-key[t, e], e))[:k] for t in range(T)])
    sel_s = np.take_along_axis(s, order, 1)
    sel_p = np.take_along_axis(p, order, 1)
    if mode == 0:
        ez = np.exp(sel_s - sel_s.max(1, keepdims=True))
        w = ez / ez.sum(1, keepdims=True)
    elif mode == 1:
        w = sel_p
    elif mode == 2:
        w = sel_p / sel_p.sum(1, keepdims=True)
    else:
        sa = 1.0 / (1.0 + np.exp(-sel_s))
        w = sa / sa.sum(1, keepdims=True)
    mask = np.ones((T, k))
    if gamma > 0:
        C = math.ceil(gamma * T * k / E)
        for e in range(E):
            rows, slots = np.nonzero(order == e)
            o = np.argsort(rows, kind="stable")
            mask[rows[o][C:], slots[o][C:]] = 0.0
    Y = np.stack([_dense_swiglu(x, Wg[e], Wu[e], Wd[e]) for e in range(E)])  # [E,T,D]
    y = np.zeros((T, x.shape[1]))
    for j in range(k):
        y += (mask[:, j] * w[:, j])[:, None] * Y[order[:, j], np.arange(T)]
    if sh:
        y += _dense_swiglu(x, sh["Ws_gate"], sh["Ws_up"], sh["Ws_down"])
    counts = np.bincount(order.ravel(), minlength=E)
    f = counts / (T * k)
    aux = 0.01 * E * float(np.sum(f * p.mean(0)))
    return dict(y=y, idx=order, w=w, dropped=(mask == 0).astype(np.uint8),
                counts=counts, aux=aux)


@pytest.mark.parametrize("mode,gamma,S", [(0, 0.0, 0), (1, 0.5, 4), (2, 1.0, 0), (0, 0.75, 6),
                                         (3, 0.0, 0), (3, 0.75, 4)])
def test_layer_against_dense_bruteforce(mode, gamma, S):
    rng = np.random.default_rng(100 + mode + S)
    T, D, E, F, k = 24, 8, 5, 6, 2
    x, Wr, Wg, Wu, Wd, sh = _rand_layer(rng, T, D, E, F, S)
    out = oracle.moe_forward(x, Wr, Wg, Wu, Wd, k=k, mode=mode, gamma=gamma,
                             alpha=0.01, **sh)
    ref = _numpy_layer(x, Wr, Wg, Wu, Wd, k, mode, gamma, sh)
    np.testing.assert_array_equal(out["idx"], ref["idx"])
    np.testing.assert_array_equal(out["dropped"], ref["dropped"])
    np.testing.assert_array_equal(out["counts"], ref["counts"])
    np.testing.assert_allclose(out["w"], ref["w"], atol=1e-12)
    np.testing.assert_allclose(out["y"], ref["y"], rtol=1e-10, atol=1e-10)
    assert abs(out["aux"] - ref["aux"]) < 1e-12
    if gamma > 0:
        assert out["dropped"].sum() > 0


def test_shared_expert_is_added_unweighted():
    rng = np.random.default_rng(31)
    x, Wr, Wg, Wu, Wd, sh = _rand_layer(rng, 20, 8, 4, 6, S=10)
    with_sh = oracle.moe_forward(x, Wr, Wg, Wu, Wd, k=2, mode=1, **sh)
    without = oracle.moe_forward(x, Wr, Wg, Wu, Wd, k=2, mode=1)
    np.testing.assert_allclose(with_sh["y"] - without["y"],
                               _dense_swiglu(x, sh["Ws_gate"], sh["Ws_up"], sh["Ws_down"]),
                               rtol=1e-10, atol=1e-10)
    # two shared experts of widths 4 and 6 equal one of width 10
    halves = [oracle.swiglu_rows(x, sh["Ws_gate"][a:b], sh["Ws_up"][a:b], sh["Ws_down"][:, a:b])
              for a, b in ((0, 4), (4, 10))]
    np.testing.assert_allclose(with_sh["y"] - without["y"], halves[0] + halves[1],
                               rtol=1e-10, atol=1e-10)


def test_dropped_top1_token_gets_shared_only():
    rng = np.random.default_rng(32)
    x, Wr, Wg, Wu, Wd, sh = _rand_layer(rng, 64, 8, 4, 6, S=5)
    out = oracle.moe_forward(x, Wr, Wg, Wu, Wd, k=1, mode=1, gamma=0.25, **sh)
    d = out["dropped"][:, 0] == 1
    assert d.sum() > 0
    sh_only = _dense_swiglu(x, sh["Ws_gate"], sh["Ws_up"], sh["Ws_down"])
    np.testing.assert_allclose(out["y"][d], sh_only[d], rtol=1e-10, atol=1e-10)


def test_expert_permutation_invariance():
    rng = np.random.default_rng(41)
    x, Wr, Wg, Wu, Wd, _ = _rand_layer(rng, 30, 8, 6, 5)
    perm = rng.permutation(6)
    a = oracle.moe_forward(x, Wr, Wg, Wu, Wd, k=3, mode=2)
    b = oracle.moe_forward(x, Wr[perm], Wg[perm], Wu[perm], Wd[perm], k=3, mode=2)
    inv = np.argsort(perm)
    np.testing.assert_array_equal(perm[b["idx"]], a["idx"])
    np.testing.assert_array_equal(b["counts"], a["counts"][perm])
    assert inv[perm[0]] == 0
    np.testing.assert_allclose(a["y"], b["y"], rtol=1e-11, atol=1e-11)


def test_sampled_rows_match_whole_layer():
    rng = np.random.default_rng(51)
    x, Wr, Wg, Wu, Wd, sh = _rand_layer(rng, 40, 8, 4, 6, S=3)
    full = oracle.moe_forward(x, Wr, Wg, Wu, Wd, k=2, mode=0, gamma=0.6, **sh)
    rows = np.array([0, 3, 17, 39])
    y = oracle.moe_rows(x[rows], full["idx"][rows], full["w"][rows], full["dropped"][rows],
                        lambda e: (Wg[e], Wu[e], Wd[e]),
                        shared=(sh["Ws_gate"], sh["Ws_up"], sh["Ws_down"]))
    np.testing.assert_allclose(y, full["y"][rows], rtol=1e-12, atol=1e-12)


def test_routing_on_given_scores():
    rng = np.random.default_rng(61)
    x, Wr, Wg, Wu, Wd, _ = _rand_layer(rng, 16, 8, 4, 6)
    s = rng.standard_normal((16, 4))
    out = oracle.moe_forward(x, Wr, Wg, Wu, Wd, k=2, mode=0, s_in=s)
    np.testing.assert_array_equal(out["s"], s)
    idx, w, _, _ = oracle.route(s, 2, 0)
    np.testing.assert_array_equal(out["idx"], idx)


# --- sigmoid gating and selection-only bias ([MPF] "The router", closing
# remark on DeepSeek-V3; [MPF] "Keeping the load even", bias balancing) ----

def test_sigmoid_gating_closed_form():
    """sigmoid(ln 9) = 0.9, sigmoid(0) = 0.5, sigmoid(ln 3) = 0.75,
    sigmoid(-ln 3) = 0.25: top-2 = experts 0 and 2 with weights 0.9/1.65 =
    6/11 and 0.75/1.65 = 5/11; P = the sigmoids over their sum 2.4."""
    s = np.array([[math.log(9.0), 0.0, math.log(3.0), -math.log(3.0)]])
    idx, w, P_sum, counts = oracle.route(s, 2, 3)
    assert idx[0].tolist() == [0, 2]
    np.testing.assert_allclose(w[0], [6 / 11, 5 / 11], rtol=0, atol=1e-14)
    np.testing.assert_allclose(P_sum, np.array([0.9, 0.5, 0.75, 0.25]) / 2.4, atol=1e-14)
    assert counts.tolist() == [1, 0, 1, 0]


def test_sigmoid_top1_weight_is_one_and_probabilities_sum_to_one():
    rng = np.random.default_rng(71)
    s = rng.standard_normal((300, 12)) * 2
    idx, w, P_sum, _ = oracle.route(s, 1, 3)
    assert np.all(w == 1.0)
    np.testing.assert_array_equal(idx[:, 0], np.argmax(s, 1))  # sigmoid is monotone
    assert abs(P_sum.sum() - 300) < 1e-9
    idx4, w4, _, _ = oracle.route(s, 4, 3)
    np.testing.assert_allclose(w4.sum(1), 1.0, atol=1e-14)


@pytest.mark.parametrize("mode", [0, 1, 2, 3])
def test_selection_bias_changes_selection_not_weights(mode):
    """A large bias forces an expert into the top k; the weights are those of
    the unbiased scores over the chosen set."""
    s = np.array([[math.log(9.0), 0.0, math.log(3.0), -math.log(3.0)]])
    b = np.array([0.0, 0.0, -10.0, 0.0], np.float32)
    idx, w, P_sum, counts = oracle.route(s, 2, mode, sel_bias=b)
    assert idx[0].tolist() == [0, 1]
    # the same set chosen without a bias, by forcing it through the scores
    # of a copy where expert 2 cannot win, gives the weights to compare
    if mode == 3:
        np.testing.assert_allclose(w[0], [0.9 / 1.4, 0.5 / 1.4], atol=1e-14)
    elif mode == 0:
        np.testing.assert_allclose(w[0], [0.9, 0.1], atol=1e-14)   # e^{ln 9}/(9 + 1)
    p = np.exp(s[0]) / np.exp(s[0]).sum()
    if mode == 1:
        np.testing.assert_allclose(w[0], p[[0, 1]], atol=1e-14)
    if mode == 2:
        np.testing.assert_allclose(w[0], p[[0, 1]] / p[[0, 1]].sum(), atol=1e-14)
    # the balance loss's probabilities ignore the bias
    _, _, P_ref, _ = oracle.route(s, 2, mode)
    np.testing.assert_allclose(P_sum, P_ref, atol=1e-15)
    assert counts.tolist() == [1, 1, 0, 0]


def test_selection_bias_constant_shift_is_neutral():
    rng = np.random.default_rng(72)
    s = np.round(rng.standard_normal((200, 8)) * 4) / 4        # dyadic: exact in fp32
    b = np.round(rng.standard_normal(8) * 4).astype(np.float32) / 4
    a = oracle.route(s, 3, 3, sel_bias=b)
    c = oracle.route(s, 3, 3, sel_bias=b + np.float32(2.0))
    for u, v in zip(a, c):
        np.testing.assert_array_equal(u, v)


@pytest.mark.parametrize("mode", [0, 3])
def test_layer_with_selection_bias_against_bruteforce(mode):
    rng = np.random.default_rng(81 + mode)
    T, D, E, F, k = 24, 8, 6, 5, 2
    x, Wr, Wg, Wu, Wd, sh = _rand_layer(rng, T, D, E, F, 3)
    b = (rng.standard_normal(E) * 0.7).astype(np.float32)
    out = oracle.moe_forward(x, Wr, Wg, Wu, Wd, k=k, mode=mode, gamma=0.8, alpha=0.01,
                             bias=b, bias_selection_only=True, **sh)
    ref = _numpy_layer(x, Wr, Wg, Wu, Wd, k, mode, 0.8, sh, sel_bias=b)
    np.testing.assert_array_equal(out["idx"], ref["idx"])
    np.testing.assert_array_equal(out["dropped"], ref["dropped"])
    np.testing.assert_array_equal(out["counts"], ref["counts"])
    np.testing.assert_allclose(out["w"], ref["w"], atol=1e-12)
    np.testing.assert_allclose(out["y"], ref["y"], rtol=1e-10, atol=1e-10)
    assert abs(out["aux"] - ref["aux"]) < 1e-12
    # the scores exclude the bias
    np.testing.assert_allclose(out["s"], x.astype(np.float64) @ Wr.astype(np.float64).T,
                               rtol=1e-12, atol=1e-12)


# --- latent MoE ([SFR], the Nemotron 3 Super variant after 'The 2026
# configuration table': x_lat = x W_in^T, the layer at width L, y = y_lat W_out^T)

def test_linear_against_matmul():
    rng = np.random.default_rng(91)
    x = rng.standard_normal((7, 13))
    W = rng.standard_normal((5, 13)).astype(np.float32)
    np.testing.assert_allclose(oracle.linear(x, W), x @ W.astype(np.float64).T,
                               rtol=1e-13, atol=1e-13)


def test_latent_with_identity_projections_is_the_plain_layer():
    rng = np.random.default_rng(92)
    x, Wr, Wg, Wu, Wd, sh = _rand_layer(rng, 30, 8, 5, 6, 4)
    eye = np.eye(8, dtype=np.float32)
    plain = oracle.moe_forward(x, Wr, Wg, Wu, Wd, k=2, mode=2, gamma=0.7, alpha=0.01, **sh)
    lat = oracle.latent_forward(x, eye, eye, Wr, Wg, Wu, Wd, k=2, mode=2, gamma=0.7,
                                alpha=0.01, **sh)
    for key in ("idx", "dropped", "counts", "kept"):
        np.testing.assert_array_equal(lat[key], plain[key])
    np.testing.assert_allclose(lat["y"], plain["y"], rtol=1e-13, atol=1e-13)
    assert abs(lat["aux"] - plain["aux"]) < 1e-15


@pytest.mark.parametrize("mode,sel", [(0, False), (3, True)])
def test_latent_against_dense_bruteforce(mode, sel):
    """x_lat = x W_in^T, the brute-force layer at width L, then y_lat W_out^T."""
    rng = np.random.default_rng(93 + mode)
    T, Do, L, E, F, k = 20, 12, 6, 5, 4, 2
    x = rng.standard_normal((T, Do)).astype(np.float32)
    W_in = (rng.standard_normal((L, Do)) / math.sqrt(Do)).astype(np.float32)
    W_out = (rng.standard_normal((Do, L)) / math.sqrt(L)).astype(np.float32)
    _, Wr, Wg, Wu, Wd, sh = _rand_layer(rng, 1, L, E, F, 3)
    b = (rng.standard_normal(E) * 0.5).astype(np.float32) if sel else None
    out = oracle.latent_forward(x, W_in, W_out, Wr, Wg, Wu, Wd, k=k, mode=mode, gamma=0.9,
                                alpha=0.01, bias=b, bias_selection_only=sel, **sh)
    x_lat = x.astype(np.float64) @ W_in.astype(np.float64).T
    ref = _numpy_layer(x_lat, Wr, Wg, Wu, Wd, k, mode, 0.9, sh, sel_bias=b)
    np.testing.assert_array_equal(out["idx"], ref["idx"])
    np.testing.assert_array_equal(out["dropped"], ref["dropped"])
    np.testing.assert_allclose(out["y"], ref["y"] @ W_out.astype(np.float64).T,
                               rtol=1e-10, atol=1e-10)
    assert abs(out["aux"] - ref["aux"]) < 1e-12


# ---------------------------------------------------------------- e4m3 weights
# The E4M3 functions are pinned against PyTorch's float8_e4m3fn type (an
# independent implementation of the same OCP format), against the format's
# own grid (every representable value encodes to itself, ties go to the even
# code), and the row quantizer against its defining properties.

def _torch_e4m3_codes(v):
    import torch
    return torch.from_numpy(np.asarray(v, dtype=np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def test_e4m3_decode_matches_torch():
    import torch
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    same = (mine == ref) | (np.isnan(mine) & np.isnan(ref))
    assert same.all()
    assert np.nanmax(mine) == 448.0 and np.isnan(mine[0x7F]) and np.isnan(mine[0xFF])
    assert mine[1] == 2.0 ** -9 and mine[8] == 2.0 ** -6   # smallest subnormal, normal


def test_e4m3_encode_matches_torch_on_grid_ties_and_random():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    # every representable value encodes to its own code (+0 and -0 distinct)
    np.testing.assert_array_equal(oracle.e4m3_encode(vals), codes)
    pos = np.sort(np.unique(oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)          # exact ties in fp32
    up = np.nextafter(mids, np.float32(np.inf))
    down = np.nextafter(mids, np.float32(-np.inf))
    rng = np.random.default_rng(5)
    rnd = (np.exp(rng.uniform(np.log(2.0 ** -12), np.log(448.0), 20000)) *
           rng.choice([-1.0, 1.0], 20000)).astype(np.float32)
    for v in (mids, -mids, up, down, rnd, np.float32([0.0, -0.0, 2.0 ** -11, -2.0 ** -10])):
        np.testing.assert_array_equal(oracle.e4m3_encode(v), _torch_e4m3_codes(v))
    # ties go to the even code (mantissa lsb 0)
    assert (oracle.e4m3_encode(mids) & 1 == 0).all()


def test_e4m3_encode_saturates():
    v = np.float32([448.0, 449.0, 463.9, 464.0, 1e6, -500.0, -1e30])
    np.testing.assert_array_equal(oracle.e4m3_encode(v),
                                  np.uint8([0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]))


def test_quantize_rows_properties():
    rng = np.random.default_rng(6)
    W = (rng.standard_normal((40, 96)) * np.exp(rng.uniform(-8, 4, (40, 1)))).astype(np.float32)
    W[3] = 0.0
    W[7, :5] = [1e-30, -1e-30, 0.0, 3.0, -3.0]
    q, s = oracle.quantize_e4m3_rows(W)
    amax = np.abs(W).max(axis=1)
    nz = amax > 0
    np.testing.assert_array_equal(s[nz], (amax[nz] / np.float32(448.0)).astype(np.float32))
    assert s[3] == 1.0 and (q[3] == 0).all()
    deq = oracle.e4m3_decode(q) * s[:, None].astype(np.float64)
    # the largest magnitude of every row lands on the largest code
    assert np.all(np.abs(oracle.e4m3_decode(q[nz])).max(axis=1) == 448.0)
    # rounding error: half a grid step of E4M3 at the value's binade
    v = W.astype(np.float64) / s[:, None]
    e = np.maximum(np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -30))), -6)
    assert np.all(np.abs(v - oracle.e4m3_decode(q)) <= 2.0 ** (e - 4) * (1 + 1e-12))
    assert np.all(np.abs(deq - W) <= np.abs(W) / 16 + s[:, None] * 2.0 ** -10 + 1e-45)


def test_swiglu_q8_equals_dense_with_dequantized_weights():
    # power-of-two scales make every dequantized weight exact in fp32, so the
    # E4M3 expert must equal the (pinned) fp32 expert on those weights
    rng = np.random.default_rng(7)
    D, F, n = 48, 40, 6
    qg = rng.integers(0, 256, (F, D), dtype=np.uint8)
    qu = rng.integers(0, 256, (F, D), dtype=np.uint8)
    qd = rng.integers(0, 256, (D, F), dtype=np.uint8)
    for q in (qg, qu, qd):
        q[(q & 0x7F) == 0x7F] = 0x40          # no NaN codes
    sg = np.float32(2.0) ** rng.integers(-12, -4, F)
    su = np.float32(2.0) ** rng.integers(-12, -4, F)
    sd = np.float32(2.0) ** rng.integers(-12, -4, D)
    x = rng.standard_normal((n, D))
    deq = lambda q, s: (oracle.e4m3_decode(q) * s[:, None]).astype(np.float32)
    got = oracle.swiglu_rows_q8(x, qg, sg, qu, su, qd, sd)
    want = oracle.swiglu_rows(x, deq(qg, sg), deq(qu, su), deq(qd, sd))
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12 * np.abs(want).max())


# ------------------------------------------------------- e4m3 activations too
def _torch_dequant_rows(v32):
    """Row-wise E4M3 round trip of fp32 rows with PyTorch's float8_e4m3fn:
    scale = max|row| / 448 in fp32 (1 for a zero row), values v / scale in
    fp32 (clamped to the format's range; the division can land a hair above
    448), cast, widened, times the scale -> fp64."""
    import torch
    v32 = np.asarray(v32, dtype=np.float32)
    amax = np.abs(v32).max(axis=1)
    s = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    q = torch.from_numpy((v32 / s[:, None]).astype(np.float32)).clamp(-448.0, 448.0)
    return q.to(torch.float8_e4m3fn).to(torch.float64).numpy() * s[:, None].astype(np.float64)


def _random_codes(rng, shape):
    q = rng.integers(0, 256, shape, dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x40              # no NaN codes
    return q


def test_swiglu_w8a8_matches_torch_float8_recomputation():
    rng = np.random.default_rng(11)
    D, F, n = 64, 48, 7
    qg, qu, qd = _random_codes(rng, (F, D)), _random_codes(rng, (F, D)), _random_codes(rng, (D, F))
    sg = (rng.uniform(0.5, 2.0, F) * 2.0 ** -9).astype(np.float32)
    su = (rng.uniform(0.5, 2.0, F) * 2.0 ** -9).astype(np.float32)
    sd = (rng.uniform(0.5, 2.0, D) * 2.0 ** -8).astype(np.float32)
    x = (rng.standard_normal((n, D)) * np.exp(rng.uniform(-3, 3, (n, 1)))).astype(np.float32)
    x[2] = 0.0                                 # a zero row: scale 1, all codes 0
    x[4, :3] = [1e-30, -200.0, 7.5]            # wide dynamic range, subnormal codes
    got = oracle.swiglu_rows_w8a8(x, qg, sg, qu, su, qd, sd)
    import torch
    deq = lambda q, s: (torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64)
                        .numpy() * s[:, None].astype(np.float64))
    Wg, Wu, Wd = deq(qg, sg), deq(qu, su), deq(qd, sd)
    xt = _torch_dequant_rows(x)
    g, u = xt @ Wg.T, xt @ Wu.T
    h32 = (g / (1.0 + np.exp(-g)) * u).astype(np.float32)
    want = _torch_dequant_rows(h32) @ Wd.T
    assert np.all(got[2] == 0.0)
    np.testing.assert_allclose(got, want, rtol=1e-9, atol=1e-9 * np.abs(want).max())
    # and the activation rounding matters: the E4M3-weight expert differs
    plain = oracle.swiglu_rows_q8(x, qg, sg, qu, su, qd, sd)
    assert np.abs(plain - got).max() > 1e-4 * np.abs(want).max()


def test_swiglu_w8a8_is_q8_expert_between_row_quantizers():
    # with W_down = I (code 0x38 = 1.0 on the diagonal, scale 1) the expert's
    # output is its dequantized hidden row, so it must equal: quantize the
    # token rows, run the (pinned) E4M3-weight expert with an identity down
    # projection, round to fp32, quantize the rows again
    rng = np.random.default_rng(12)
    D = F = 40
    n = 9
    qg, qu = _random_codes(rng, (F, D)), _random_codes(rng, (F, D))
    sg = (2.0 ** rng.integers(-10, -6, F)).astype(np.float32)
    su = (rng.uniform(0.5, 2.0, F) * 2.0 ** -8).astype(np.float32)
    qd = np.zeros((D, F), dtype=np.uint8)
    np.fill_diagonal(qd, 0x38)
    sd = np.ones(D, dtype=np.float32)
    assert oracle.e4m3_decode(np.uint8([0x38]))[0] == 1.0
    x = (rng.standard_normal((n, D)) * 3.0).astype(np.float32)
    got = oracle.swiglu_rows_w8a8(x, qg, sg, qu, su, qd, sd)

    def round_trip(v):
        q, s = oracle.quantize_e4m3_rows(np.asarray(v, dtype=np.float32))
        return oracle.e4m3_decode(q) * s[:, None].astype(np.float64)

    h = oracle.swiglu_rows_q8(round_trip(x), qg, sg, qu, su, qd, sd)
    np.testing.assert_array_equal(got, round_trip(h.astype(np.float32)))
