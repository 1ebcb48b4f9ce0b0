"""Calls from several host threads at once (GPU).

Each thread drives its own layer shape on its own stream with its own
outputs and workspace; the first calls of a fresh process race through the
library's one-time per-device launch setup.  The kernels are deterministic
(no atomics on the data path, fixed summation orders), so every thread's
result must equal, bit for bit, the same call made afterwards on one thread.
Runs in a child process so that nothing is set up before the threads start."""
import os
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent(r"""
    import sys, threading
    import torch
    sys.path.insert(0, sys.argv[1])
    from mixture_experts_layer_capacity_b300 import binding as B
    from mixture_experts_layer_capacity_b300.workloads import Workload, make_inputs

    shapes = [
        # Switch-like: fused router, capacity drops, down GEMM writing y
        Workload("t_switch", T=1024, D=512, E=8, F=1024, k=1, mode=1, gamma=1.0,
                 bias="normal_var2"),
        # top-2 with a shared expert whose tiles join the routed launches
        Workload("t_shared", T=300, D=256, E=8, F=512, k=2, mode=0, S=1024),
        # many experts, renormalised weights, tensor-core router
        Workload("t_wide", T=777, D=256, E=64, F=256, k=6, mode=2, gamma=1.25,
                 bias="zipf1.1"),
    ]
    dev = torch.device("cuda", 0)
    jobs = []
    for i, w in enumerate(shapes):
        cfg = B.config_of(w)
        inputs = make_inputs(w, 100 + i, dev)
        jobs.append((cfg, inputs, B.alloc_outputs(cfg, dev), torch.cuda.Stream(dev)))
    torch.cuda.synchronize()

    start = threading.Barrier(len(jobs))
    errors = []

    def run(job):
        cfg, inputs, outs, stream = job
        try:
            start.wait()
            for _ in range(20):
                B.forward(cfg, inputs, outs, stream=stream)
            stream.synchronize()
        except Exception as exc:  # reported by the main thread
            errors.append(repr(exc))

    threads = [threading.Thread(target=run, args=(j,)) for j in jobs]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in threads), "a thread did not finish"
    assert not errors, errors

    keys = ["y", "router_logits", "topk_idx", "topk_w", "dropped_mask", "expert_counts",
            "kept_counts", "aux_loss"]
    for cfg, inputs, outs, _ in jobs:
        assert B.read_device_status(cfg, outs["workspace"]) == B.MOE_DEVICE_OK
        ref = B.forward(cfg, inputs)
        torch.cuda.synchronize()
        for k in keys:
            assert torch.equal(outs[k], ref[k]), (cfg.T, k)
    print("threads ok", len(jobs))
""")


@pytest.mark.gpu
def test_concurrent_calls_from_host_threads():
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "threads ok 3" in r.stdout
