"""One batch split over several ranks (moe_sharded_route / moe_sharded_finish)
against the CPU oracle run on the WHOLE batch, through the C ABI.

The ranks are emulated one after another on one GPU: each rank's route call,
then the exchange (the per-rank counts and sums stacked in rank order, which
is what the all-gather of sharded.gather_rank_stats produces), then each
rank's finish call.  No kernel waits on another rank's kernels.  The
concatenated per-rank outputs must pass every parity criterion of a single
call over the batch: capacity drops in global token order, demand and kept
counts summed over ranks, and the balance loss of the whole batch."""
import numpy as np
import pytest
import torch

import oracle
import parity
from mixture_experts_layer_capacity_b300 import binding as B
from mixture_experts_layer_capacity_b300 import sharded
from mixture_experts_layer_capacity_b300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu

# name, T, D, E, F, k, S, mode, gamma, bias, dtype, token counts per rank
CASES = [
    ("two_ranks_top2_capacity", 1000, 256, 8, 384, 2, 192, 0, 0.75, "normal_var2", "bf16",
     [500, 500]),
    ("three_ranks_e64_drops", 900, 128, 64, 128, 8, 0, 2, 1.0, "zipf1.1", "bf16",
     [300, 300, 300]),
    ("uneven_with_empty_rank", 777, 192, 16, 320, 4, 0, 1, 0.75, "normal_var2", "bf16",
     [0, 500, 1, 276]),
    ("four_ranks_top1_direct_y", 1536, 256, 8, 256, 1, 0, 1, 0.5, "normal_var2", "bf16",
     [384, 384, 384, 384]),
    ("two_ranks_dropless_shared", 640, 128, 8, 192, 2, 128, 0, 0.0, "none", "bf16",
     [320, 320]),
    ("two_ranks_fp32", 300, 64, 8, 64, 2, 32, 1, 0.75, "normal_var2", "fp32", [173, 127]),
]


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    torch.cuda.synchronize()


def _run_ranks(w, inp, counts, tamper=None):
    """Route, exchange and finish for every rank; returns (cfgs, outs, slices)."""
    T = w.T
    assert sum(counts) == T
    starts = np.concatenate([[0], np.cumsum(counts)[:-1]]).astype(int)
    cfgs, outs, views = [], [], []
    for s, n in zip(starts, counts):
        cfg = B.make_config(n, w.D, w.E, w.F, w.k, w.S, w.dtype, w.mode, w.gamma, w.alpha,
                            bias_selection_only=w.sel_bias)
        v = dict(inp)
        v["x"] = inp["x"][int(s):int(s) + int(n)]
        o = sharded.alloc_outputs(cfg, T, "cuda")
        sharded.route(cfg, T, v, o)
        cfgs.append(cfg)
        outs.append(o)
        views.append(v)
    all_c = torch.stack([o["expert_counts"] for o in outs]).contiguous()
    all_p = torch.stack([o["prob_sums"] for o in outs]).contiguous()
    if tamper is not None:
        tamper(all_c)
    for r, (cfg, o, v) in enumerate(zip(cfgs, outs, views)):
        sharded.finish(cfg, T, len(counts), r, all_c, all_p, v, o)
    return cfgs, outs, list(zip(starts, counts))


def _concat(outs):
    cat = lambda key: torch.cat([o[key] for o in outs], 0)
    return dict(
        router_logits=cat("router_logits"), topk_idx=cat("topk_idx"), topk_w=cat("topk_w"),
        dropped_mask=cat("dropped_mask"), y=cat("y"),
        expert_counts=torch.stack([o["expert_counts"] for o in outs]).sum(0),
        kept_counts=torch.stack([o["kept_counts"] for o in outs]).sum(0),
        aux_loss=outs[0]["aux_loss"])


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_split_batch_matches_whole_batch(case):
    name, T, D, E, F, k, S, mode, gamma, bias, dtype, counts = case
    w = Workload(name, T=T, D=D, E=E, F=F, k=k, S=S, mode=mode, gamma=gamma, dtype=dtype,
                 alpha=0.01, bias=bias)
    inp = make_inputs(w, 21, "cuda")
    cfgs, outs, slices = _run_ranks(w, inp, counts)
    for cfg, o in zip(cfgs, outs):
        assert B.read_device_status(cfg, o["workspace"]) == B.MOE_DEVICE_OK
    # every rank reports the loss of the whole batch, bit for bit the same
    auxes = {float(o["aux_loss"][0]) for o in outs}
    assert len(auxes) == 1, auxes
    full = _concat(outs)
    rep = parity.check(w, inp, full)
    # per rank: its own demand counts, and kept counts that follow the
    # whole-batch drops of its rows
    idx = full["topk_idx"].cpu().numpy()
    dropped = full["dropped_mask"].cpu().numpy()
    for (s, n), o in zip(slices, outs):
        ii, dd = idx[s:s + n], dropped[s:s + n]
        want_n = np.bincount(ii.ravel(), minlength=E)
        want_kept = np.bincount(ii[dd == 0].ravel(), minlength=E)
        np.testing.assert_array_equal(o["expert_counts"].cpu().numpy(), want_n)
        np.testing.assert_array_equal(o["kept_counts"].cpu().numpy(), want_kept)
    if gamma > 0:
        # the capacity is the whole batch's, and the split moved no drop
        C = oracle.capacity(T, k, E, float(np.float32(gamma)))
        assert int(full["kept_counts"].max()) <= C
    print(name, rep)


def test_exchanged_counts_are_checked():
    """Counts that do not add up to T_global * k are refused by the kernel
    (status word), and the later kernels skip their work."""
    w = Workload("tamper", T=600, D=128, E=8, F=128, k=2, S=0, mode=0, gamma=1.0,
                 dtype="bf16", alpha=0.01)
    inp = make_inputs(w, 22, "cuda")

    def tamper(all_c):
        all_c[0, 0] += 1

    cfgs, outs, _ = _run_ranks(w, inp, [300, 300], tamper=tamper)
    for cfg, o in zip(cfgs, outs):
        assert B.read_device_status(cfg, o["workspace"]) == B.MOE_DEVICE_SHARD_MISMATCH



def _corrupt_last_token(outs, rank, E, how):
    """Gives the last token of `rank` an expert index the finish launch must
    refuse: one outside [0, E) ("range"), or a valid expert that does not
    occur among the rank's last 32 tokens ("segment": that token's row would
    then fall past the expert's segment, since every routing-kernel block
    holds at most 32 tokens at these sizes)."""
    idx = outs[rank]["topk_idx"]
    last = idx[-1].clone()
    if how == "range":
        idx[-1, 0] = E + 3
        return
    recent = set(idx[-32:].flatten().tolist())
    spare = [e for e in range(E) if e not in recent]
    assert spare, "every expert occurs among the last 32 tokens"
    idx[-1, 0] = spare[0]
    assert not torch.equal(idx[-1], last)


@pytest.mark.parametrize("how", ["range", "segment"])
def test_finish_refuses_bad_expert_indices(how):
    """moe_sharded_finish reads topk_idx as the caller hands it back.  An
    index outside [0, E), or one whose row would fall outside its expert's
    segment, is refused by the kernel's own check (status word, no access),
    and the next normal split call on the same workspaces is correct."""
    w = Workload("bad_idx", T=800, D=128, E=64, F=128, k=2, S=0, mode=2, gamma=0.0,
                 dtype="bf16", alpha=0.01, bias="zipf1.1")
    inp = make_inputs(w, 23, "cuda")
    counts = [400, 400]
    T = w.T
    starts = [0, 400]
    cfgs, outs, views = [], [], []
    for s, n in zip(starts, counts):
        cfg = B.make_config(n, w.D, w.E, w.F, w.k, w.S, w.dtype, w.mode, w.gamma, w.alpha)
        v = dict(inp)
        v["x"] = inp["x"][s:s + n]
        o = sharded.alloc_outputs(cfg, T, "cuda")
        sharded.route(cfg, T, v, o)
        cfgs.append(cfg)
        outs.append(o)
        views.append(v)
    all_c = torch.stack([o["expert_counts"] for o in outs]).contiguous()
    all_p = torch.stack([o["prob_sums"] for o in outs]).contiguous()
    torch.cuda.synchronize()
    _corrupt_last_token(outs, 1, w.E, how)
    for r in range(2):
        sharded.finish(cfgs[r], T, 2, r, all_c, all_p, views[r], outs[r])
    assert B.read_device_status(cfgs[0], outs[0]["workspace"]) == B.MOE_DEVICE_OK
    assert B.read_device_status(cfgs[1], outs[1]["workspace"]) == \
        B.MOE_DEVICE_INDEX_OUT_OF_RANGE
    # the same workspaces, a clean split call: the whole-batch oracle again
    cfgs2, outs2, _ = _run_ranks(w, inp, counts)
    for cfg, o in zip(cfgs2, outs2):
        assert B.read_device_status(cfg, o["workspace"]) == B.MOE_DEVICE_OK
    parity.check(w, inp, _concat(outs2))
