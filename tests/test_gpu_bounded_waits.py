"""The bounded waits, exercised on the GPU in a form that faults nothing.

Every wait in the library's kernels gives up after a time limit, records
MOE_DEVICE_PIPELINE_TIMEOUT in the status word and lets the kernel return;
the later kernels of the forward pass see the status and do no work.  The
test hook moe_debug_barrier_fault makes the routing kernel's grid-wide
barrier wait for one block more than the grid has (so it can never
complete) with a 1 ms limit.  No copy or other asynchronous work is in
flight at that barrier.  The test checks that the forward pass returns with
the timeout status within a fraction of the default 2 s limit, and that the
next normal call on the same context matches the oracle."""
import time

import pytest
import torch

import parity
from mixture_experts_layer_capacity_b300 import binding as B
from mixture_experts_layer_capacity_b300.workloads import WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu

CASES = [
    # bf16, router fused into the routing kernel, capacity drops, shared expert
    Workload("timeout_fused_router", T=640, D=256, E=8, F=256, k=2, S=128, mode=0,
             gamma=1.0, dtype="bf16"),
    # bf16, tensor-core router GEMM before the routing kernel, 64 experts
    Workload("timeout_tc_router", T=1024, D=512, E=64, F=128, k=8, S=0, mode=2,
             gamma=0.0, dtype="bf16", bias="zipf1.1"),
    WORKLOADS["tiny_fp32"],
]


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    B.debug_barrier_fault(0, 0)
    torch.cuda.synchronize()


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_barrier_timeout_sets_status_and_the_next_call_is_normal(w):
    cfg = B.config_of(w)
    inp = make_inputs(w, 21, "cuda")
    outs = B.alloc_outputs(cfg)
    torch.cuda.synchronize()
    B.debug_barrier_fault(1, 1_000_000)           # one arrival too many, 1 ms limit
    try:
        t0 = time.perf_counter()
        B.forward(cfg, inp, outs)
        code = B.read_device_status(cfg, outs["workspace"])
        dt = time.perf_counter() - t0
    finally:
        B.debug_barrier_fault(0, 0)
    assert code == B.MOE_DEVICE_PIPELINE_TIMEOUT
    assert dt < 1.0, dt                            # the 1 ms limit, not the 2 s default
    # the same context, the same workspace: a normal call matches the oracle
    B.forward(cfg, inp, outs)
    assert B.read_device_status(cfg, outs["workspace"]) == B.MOE_DEVICE_OK
    print(w.name, f"timed out in {dt * 1e3:.1f} ms;", parity.check(w, inp, outs))
