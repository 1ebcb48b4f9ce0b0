"""One batch of tokens split over the ranks of a ``torch.distributed`` group
(data parallel), with the same results as one layer call over the whole batch.

Capacity is applied in token order over the whole batch ("Mixture of Experts"
(module 17), 17.5) and the balance loss uses f_e and P_e over the whole batch
(17.4), so the ranks exchange, once per layer, their per-expert demand counts
and probability sums.  Per rank (ranks hold consecutive token ranges, in rank
order):

  1. ``moe_sharded_route`` gates the rank's tokens and writes its counts and sums;
  2. ``gather_rank_stats`` all-gathers them in rank order (the exchange);
  3. ``moe_sharded_finish`` keeps an assignment iff (assignments of earlier
     ranks to its expert) + (its position on this rank) < C, then runs the
     experts, the combine and the balance loss over all ranks.

Everything but the all-gather runs in libmoe's kernels; this module only
allocates, slices and calls.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import binding as B


def token_slices(T_global: int, n_ranks: int):
    """(start, count) of each rank's tokens: consecutive ranges in rank order,
    the first T_global % n_ranks ranks one token longer."""
    base, extra = divmod(int(T_global), int(n_ranks))
    out, start = [], 0
    for r in range(n_ranks):
        n = base + (1 if r < extra else 0)
        out.append((start, n))
        start += n
    return out


def gather_rank_stats(expert_counts: torch.Tensor, prob_sums: torch.Tensor, group=None):
    """All-gather of every rank's demand counts [E] (int32) and probability
    sums [E] (fp64) into [n_ranks, E] tensors, row r = rank r.  Works on CUDA
    tensors (NCCL) and CPU tensors (gloo)."""
    world = dist.get_world_size(group)
    E = int(expert_counts.numel())
    all_c = torch.empty((world, E), dtype=expert_counts.dtype, device=expert_counts.device)
    all_p = torch.empty((world, E), dtype=prob_sums.dtype, device=prob_sums.device)
    dist.all_gather(list(all_c.unbind(0)), expert_counts.contiguous(), group=group)
    dist.all_gather(list(all_p.unbind(0)), prob_sums.contiguous(), group=group)
    return all_c, all_p


def alloc_outputs(cfg: B.MoeConfig, T_global: int, device="cuda"):
    """Outputs of one rank (cfg.T = its tokens) plus prob_sums [E] fp64 and
    the split-batch workspace."""
    outs = B.alloc_outputs(cfg, device)
    ws = B.sharded_workspace_size(cfg, T_global)
    outs["workspace"] = torch.empty((max(ws, 256),), dtype=torch.uint8, device=device)
    outs["prob_sums"] = torch.empty((cfg.n_experts,), dtype=torch.float64, device=device)
    return outs


def route(cfg: B.MoeConfig, T_global: int, inputs: dict, outs: dict, stream=None) -> None:
    """Step 1 on this rank's inputs (x holds the rank's tokens)."""
    B.moe_sharded_route(cfg, T_global, inputs["x"], inputs["W_r"], inputs.get("b_r"),
                        outs["router_logits"], outs["topk_idx"], outs["topk_w"],
                        outs["expert_counts"], outs["prob_sums"], outs["workspace"],
                        stream=stream)


def finish(cfg: B.MoeConfig, T_global: int, n_ranks: int, rank: int, all_counts, all_psum,
           inputs: dict, outs: dict, stream=None) -> None:
    """Step 3, given the gathered [n_ranks, E] counts and sums."""
    B.moe_sharded_finish(cfg, T_global, n_ranks, rank, all_counts, all_psum, inputs["x"],
                         inputs["W_gate"], inputs["W_up"], inputs["W_down"],
                         inputs.get("Ws_gate"), inputs.get("Ws_up"), inputs.get("Ws_down"),
                         outs["topk_idx"], outs["topk_w"], outs["y"], outs["dropped_mask"],
                         outs["kept_counts"], outs["aux_loss"], outs["workspace"],
                         stream=stream)


def forward(cfg: B.MoeConfig, T_global: int, inputs: dict, outs: dict | None = None,
            group=None) -> dict:
    """The layer on this rank's share of a batch split over ``group``.
    ``cfg.T`` and ``inputs["x"]`` hold this rank's tokens (see token_slices);
    all calls run on torch's current stream, where the collective runs too."""
    if outs is None:
        outs = alloc_outputs(cfg, T_global, inputs["x"].device)
    route(cfg, T_global, inputs, outs)
    all_c, all_p = gather_rank_stats(outs["expert_counts"], outs["prob_sums"], group)
    finish(cfg, T_global, dist.get_world_size(group), dist.get_rank(group), all_c, all_p,
           inputs, outs)
    return outs
