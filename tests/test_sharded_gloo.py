"""The split-batch exchange on CPU ranks (gloo, world size 2).

Each rank gates its own token range with the oracle (standing in for the
route kernel, which needs a GPU), exchanges its per-expert demand counts and
probability sums with ``sharded.gather_rank_stats`` (the library's one
collective), and applies the rule the finish kernel implements: an
assignment is kept iff (earlier ranks' assignments to its expert) + (its
position on this rank) < C of the whole batch.  The result must equal the
oracle's capacity over the WHOLE batch on this rank's rows, and the balance
loss from the exchanged sums must equal the whole batch's."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from mixture_experts_layer_capacity_b300 import sharded
from mixture_experts_layer_capacity_b300.workloads import Workload, make_inputs

CASES = [
    # T, D, E, k, mode, gamma, bias
    (601, 64, 8, 2, 0, 0.75, "normal_var2"),
    (300, 32, 16, 4, 2, 1.0, "zipf1.1"),
    (257, 32, 4, 1, 1, 0.5, "normal_var2"),
]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _whole_batch(case):
    T, D, E, k, mode, gamma, bias = case
    w = Workload("gloo", T=T, D=D, E=E, F=64, k=k, mode=mode, gamma=gamma, dtype="fp32",
                 alpha=0.01, bias=bias)
    inp = make_inputs(w, 31, "cpu", weights=False)
    x = inp["x"].numpy()
    b = None if inp["b_r"] is None else inp["b_r"].numpy()
    s = oracle.router_logits(x, inp["W_r"].numpy(), b)
    return w, s


def _rank_main(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out = []
        for case in CASES:
            w, s = _whole_batch(case)
            T, E, k = w.T, w.E, w.k
            start, n = sharded.token_slices(T, world)[rank]
            # this rank's gating (oracle in place of the route kernel)
            idx, _, P_sum, counts = oracle.route(s[start:start + n], k, w.mode)
            all_c, all_p = sharded.gather_rank_stats(
                torch.as_tensor(counts.astype(np.int32)), torch.as_tensor(P_sum), None)
            all_c, all_p = all_c.numpy(), all_p.numpy()
            # rank order: row r is rank r's own statistics
            for r, (s0, n0) in enumerate(sharded.token_slices(T, world)):
                _, _, P_r, c_r = oracle.route(s[s0:s0 + n0], k, w.mode)
                assert np.array_equal(all_c[r], c_r.astype(np.int32)), (rank, r)
                assert np.array_equal(all_p[r], P_r), (rank, r)
            # the finish kernel's rule, from the exchanged counts only
            C = oracle.capacity(T, k, E, float(np.float32(w.gamma)))
            before = all_c[:rank].sum(0)
            pos = np.zeros(E, np.int64)
            dropped = np.zeros((n, k), np.uint8)
            for t in range(n):
                for j in range(k):
                    e = idx[t, j]
                    dropped[t, j] = 0 if C < 0 or before[e] + pos[e] < C else 1
                    pos[e] += 1
            # the whole batch, by the oracle
            idx_all, _, P_all, counts_all = oracle.route(s, k, w.mode)
            drop_all, _ = oracle.apply_capacity(idx_all, E, C)
            assert np.array_equal(idx, idx_all[start:start + n])
            assert np.array_equal(dropped, drop_all[start:start + n]), rank
            assert np.array_equal(all_c.sum(0), counts_all)
            aux_split = oracle.aux_loss(T, k, E, float(np.float32(w.alpha)),
                                        all_c.sum(0).astype(np.int64), all_p.sum(0))
            aux_all = oracle.aux_loss(T, k, E, float(np.float32(w.alpha)), counts_all, P_all)
            assert abs(aux_split - aux_all) <= 1e-12 * abs(aux_all)
            out.append(int(dropped.sum()))
        results[rank] = out
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_rank_exchange_reproduces_whole_batch_capacity():
    world = 2
    ctx = mp.get_context("spawn")
    results = ctx.Manager().dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), results), nprocs=world,
                       join=True, start_method="spawn")
    assert sorted(results.keys()) == [0, 1]
    # drops happen on the ranks (the cases overload some experts)
    assert sum(sum(v) for v in results.values()) > 0


def test_token_slices():
    assert sharded.token_slices(10, 3) == [(0, 4), (4, 3), (7, 3)]
    assert sharded.token_slices(2, 4) == [(0, 1), (1, 1), (2, 0), (2, 0)]
    assert sharded.token_slices(0, 2) == [(0, 0), (0, 0)]


def _plumbing_main(rank, world, port, results):
    """sharded.forward on CPU tensors with the library's two calls replaced
    by recorders: the exchange between them must hand every rank's counts and
    sums, in rank order, to the finish call of every rank."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from mixture_experts_layer_capacity_b300 import binding as B
        E, T_global = 8, 37
        start, n = sharded.token_slices(T_global, world)[rank]
        cfg = B.make_config(n, 64, E, 64, 2)
        calls = {}

        def fake_route(cfg_, T_g, x, W_r, bias, logits, idx, w, counts, psum, ws, **kw):
            calls["route"] = (int(cfg_.T), int(T_g), tuple(x.shape))
            counts.copy_(torch.arange(E, dtype=torch.int32) + 100 * rank)
            psum.copy_(torch.full((E,), 0.5 + rank, dtype=torch.float64))

        def fake_finish(cfg_, T_g, n_ranks, r, all_c, all_p, *rest, **kw):
            calls["finish"] = (int(T_g), int(n_ranks), int(r), all_c.clone(), all_p.clone())

        B.moe_sharded_route = fake_route
        B.moe_sharded_finish = fake_finish
        inputs = {"x": torch.zeros((n, 64)), "W_r": None, "W_gate": None, "W_up": None,
                  "W_down": None}
        sharded.forward(cfg, T_global, inputs)
        assert calls["route"] == (n, T_global, (n, 64))
        T_g, n_ranks, r, all_c, all_p = calls["finish"]
        assert (T_g, n_ranks, r) == (T_global, world, rank)
        for rr in range(world):
            assert torch.equal(all_c[rr], torch.arange(E, dtype=torch.int32) + 100 * rr)
            assert torch.all(all_p[rr] == 0.5 + rr)
        results[rank] = True
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_sharded_forward_plumbing():
    world = 2
    ctx = mp.get_context("spawn")
    results = ctx.Manager().dict()
    mp.start_processes(_plumbing_main, args=(world, _free_port(), results), nprocs=world,
                       join=True, start_method="spawn")
    assert dict(results) == {0: True, 1: True}
