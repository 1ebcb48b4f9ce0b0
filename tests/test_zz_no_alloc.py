"""moe_forward_no_alloc against moe_forward, through the C ABI.

moe_forward_no_alloc serves callers that cannot allocate device memory (a
program with no device allocator of its own, or a serving loop that must not
call cudaMalloc): it runs the same layer with the library's static device
scratch instead of a caller workspace.  Its outputs must match the existing
entry point's, on two calls in a row (the scratch keeps the previous call's
contents, which must not leak into the next call); the two entry points run
the same kernels, so the outputs must be bit-identical.  This file is collected
last so that a run stopping at the first failure has run every other test.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_capacity_b300 import binding as B
from mixture_experts_layer_capacity_b300.workloads import WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu

CASES = [
    WORKLOADS["switch_top1_capacity"],   # k = 1, drops, down projection writes y
    WORKLOADS["tiny_fp32"],
    Workload("shared_top2", T=700, D=256, E=8, F=384, k=2, S=192, mode=0, gamma=1.25,
             dtype="bf16", bias="normal_var2"),
]


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    torch.cuda.synchronize()


def _no_alloc(cfg, inp):
    outs = B.alloc_outputs(cfg)
    del outs["workspace"]
    B.moe_forward_no_alloc(cfg, inp["x"], inp["W_r"], inp.get("b_r"), inp["W_gate"],
                           inp["W_up"], inp["W_down"], inp.get("Ws_gate"), inp.get("Ws_up"),
                           inp.get("Ws_down"), outs["y"], outs["router_logits"],
                           outs["topk_idx"], outs["topk_w"], outs["dropped_mask"],
                           outs["expert_counts"], outs["kept_counts"], outs["aux_loss"])
    torch.cuda.synchronize()
    return outs


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_matches_moe_forward_on_two_calls(w):
    cfg = B.config_of(w)
    assert B.workspace_size(cfg) <= B.STATIC_SCRATCH_BYTES
    inp = make_inputs(w, 11, "cuda")
    ref = B.forward(cfg, inp)
    torch.cuda.synchronize()
    # the same kernels on the same inputs: every output is bit-identical
    # (the library's results do not vary from run to run on one device)
    for _ in range(2):
        got = _no_alloc(cfg, inp)
        for key in ("y", "router_logits", "topk_idx", "topk_w", "dropped_mask",
                    "expert_counts", "kept_counts", "aux_loss"):
            assert torch.equal(got[key], ref[key]), key


def test_rejects_layers_larger_than_the_static_scratch():
    w = WORKLOADS["mixtral_prefill"]
    cfg = B.config_of(w)
    assert B.workspace_size(cfg) > B.STATIC_SCRATCH_BYTES
    # the size check comes before any launch; these pointers are never touched
    fake = [256 * (i + 1) for i in range(17)]
    with pytest.raises(B.MoeError) as ei:
        B.moe_forward_no_alloc(cfg, *fake)
    assert ei.value.status == B.MOE_ERR_WORKSPACE
    assert np.isfinite(B.workspace_size(cfg))
