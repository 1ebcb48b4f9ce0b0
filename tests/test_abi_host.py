"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point include/moe.h declares, and validates its arguments and
computes the capacity on the host before touching the device."""
import ctypes
import glob
import os
import re

import numpy as np
import pytest

import oracle
from conftest import ROOT
from mixture_experts_layer_capacity_b300 import binding as B
from mixture_experts_layer_capacity_b300.workloads import WORKLOADS


def _declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        txt = open(h).read()
        names |= set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", txt))
    return sorted(names)


def test_library_exports_every_declared_symbol():
    names = _declared_symbols()
    assert "moe_forward" in names and len(names) >= 5
    L = B.lib()
    for n in names:
        assert hasattr(L, n), f"libmoe.so does not export {n}"


def test_no_internal_symbols_leak():
    out = os.popen(f"nm -D --defined-only {B.LIB_PATH}").read().split("\n")
    exported = [l.split()[-1] for l in out if " T " in l]
    assert all(n.startswith("moe_") for n in exported), exported


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_capacity_matches_oracle(name):
    w = WORKLOADS[name]
    cfg = B.config_of(w)
    want = oracle.capacity(w.T, w.k, w.E, float(np.float32(w.gamma)))
    assert B.capacity(cfg) == want


@pytest.mark.parametrize("T,k,E,gamma", [(4096, 8, 64, 1.25), (4096, 1, 8, 1.0),
                                         (1000, 2, 7, 1.1), (33, 3, 5, 0.3), (1, 1, 8, 2.0),
                                         (100, 2, 4, 0.0), (100, 2, 4, -3.0)])
def test_capacity_formula(T, k, E, gamma):
    cfg = B.make_config(T, 64, E, 64, k, capacity_factor=gamma)
    assert B.capacity(cfg) == oracle.capacity(T, k, E, float(np.float32(gamma)))


def test_capacity_beyond_int64_saturates():
    """A capacity factor so large that ceil(gamma*T*k/E) leaves int64 keeps
    every assignment: library and oracle both report INT64_MAX, and the
    scratch is that of a layer that drops nothing."""
    big = B.make_config(4096, 512, 8, 2048, 2, capacity_factor=3.0e38)
    assert B.capacity(big) == 2**63 - 1 == oracle.capacity(4096, 2, 8, 3.0e38)
    roomy = B.make_config(4096, 512, 8, 2048, 2, capacity_factor=8.0)   # C = 8192 = T*k
    assert B.capacity(roomy) == 4096 * 2
    assert B.workspace_size(big) == B.workspace_size(roomy)
    idx = np.random.default_rng(0).integers(0, 8, size=(64, 2)).astype(np.int32)
    dropped, kept = oracle.apply_capacity(idx, 8, 2**63 - 1)
    assert not dropped.any() and kept.sum() == 128


def test_widths_beyond_two_to_the_twenty_are_unsupported():
    """Widths are bounded so that no workspace term can leave size_t."""
    w = 1 << 20
    ok = B.make_config(64, w, 8, 64, 2)
    assert B.workspace_size(ok) > 0
    for cfg in (B.make_config(64, w + 64, 8, 64, 2), B.make_config(64, 64, 8, w + 64, 2),
                B.make_config(64, 64, 8, 64, 2, d_shared=w + 64)):
        n = ctypes.c_size_t(0)
        assert B.lib().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == \
            B.MOE_ERR_UNSUPPORTED
    n = ctypes.c_size_t(0)
    small = B.make_config(64, 64, 8, 64, 2)
    assert B.lib().moe_latent_workspace_size(ctypes.byref(small), w + 64, ctypes.byref(n)) == \
        B.MOE_ERR_UNSUPPORTED
    assert B.lib().moe_latent_workspace_size(ctypes.byref(small), w, ctypes.byref(n)) == B.MOE_OK


def test_workspace_size_and_validation():
    ok = B.make_config(4096, 512, 8, 2048, 1, capacity_factor=1.0)
    n1 = B.workspace_size(ok)
    assert n1 > 0
    # more tokens never need less scratch
    assert B.workspace_size(B.make_config(8192, 512, 8, 2048, 1, capacity_factor=1.0)) >= n1
    bad = [
        (dict(T=-1), B.MOE_ERR_INVALID_ARG),
        (dict(top_k=0), B.MOE_ERR_INVALID_ARG),
        (dict(top_k=9, n_experts=16), B.MOE_ERR_UNSUPPORTED),
        (dict(top_k=3, n_experts=2), B.MOE_ERR_INVALID_ARG),
        (dict(n_experts=257), B.MOE_ERR_UNSUPPORTED),
        (dict(d_model=100), B.MOE_ERR_UNSUPPORTED),     # bf16 needs multiples of 64
        (dict(d_expert=96), B.MOE_ERR_UNSUPPORTED),
        (dict(d_shared=32), B.MOE_ERR_UNSUPPORTED),
        (dict(gating_mode=4), B.MOE_ERR_INVALID_ARG),
        (dict(gating_mode=-1), B.MOE_ERR_INVALID_ARG),
        (dict(dtype=7), B.MOE_ERR_INVALID_ARG),
        (dict(capacity_factor=float("nan")), B.MOE_ERR_INVALID_ARG),
    ]
    base = dict(T=64, d_model=128, n_experts=8, d_expert=128, top_k=2)
    for over, code in bad:
        kw = dict(base)
        kw.update(over)
        cfg = B.make_config(**kw)
        with pytest.raises(B.MoeError) as ei:
            B.workspace_size(cfg)
        assert ei.value.status == code, over
    # fp32 accepts any sizes
    assert B.workspace_size(B.make_config(10, 5, 3, 7, 2, dtype="fp32")) > 0
    # the sigmoid mode and the selection-only bias flag (0 or 1)
    assert B.workspace_size(B.make_config(64, 128, 8, 128, 2, gating_mode=3,
                                          bias_selection_only=True)) > 0
    cfg = B.make_config(64, 128, 8, 128, 2)
    cfg.bias_selection_only = 2
    with pytest.raises(B.MoeError) as ei:
        B.workspace_size(cfg)
    assert ei.value.status == B.MOE_ERR_INVALID_ARG


def _call(cfg, ptrs, ws_bytes):
    L = B.lib()
    args = [ptrs.get(n) for n in ("x", "W_r", "b", "Wg", "Wu", "Wd", "Wsg", "Wsu", "Wsd", "y",
                                  "logits", "idx", "w", "drop", "cnt", "kept", "aux", "ws")]
    return L.moe_forward(ctypes.byref(cfg), *args, ctypes.c_size_t(ws_bytes), None)


def test_forward_rejects_bad_arguments_before_launching():
    cfg = B.make_config(64, 128, 8, 128, 2, d_shared=128)
    need = B.workspace_size(cfg)
    fake = {n: 4096 * (i + 1) for i, n in enumerate(
        ("x", "W_r", "Wg", "Wu", "Wd", "Wsg", "Wsu", "Wsd", "y", "logits", "idx", "w",
         "drop", "cnt", "kept", "aux"))}
    fake["ws"] = 1 << 20
    # a missing output
    p = dict(fake)
    p["y"] = None
    assert _call(cfg, p, need) == B.MOE_ERR_INVALID_ARG
    # shared expert declared but its weights missing
    p = dict(fake)
    p["Wsd"] = None
    assert _call(cfg, p, need) == B.MOE_ERR_INVALID_ARG
    # workspace too small / misaligned / missing
    assert _call(cfg, fake, need - 1) == B.MOE_ERR_WORKSPACE
    p = dict(fake)
    p["ws"] = (1 << 20) + 128
    assert _call(cfg, p, need) == B.MOE_ERR_WORKSPACE
    p["ws"] = None
    assert _call(cfg, p, need) == B.MOE_ERR_WORKSPACE
    # bf16 tensors must be 16-byte aligned (tensor-map bases)
    p = dict(fake)
    p["x"] = 4096 + 8
    assert _call(cfg, p, need) == B.MOE_ERR_INVALID_ARG
    # invalid config
    bad = B.make_config(64, 128, 8, 128, 0)
    assert _call(bad, fake, need) == B.MOE_ERR_INVALID_ARG


def test_status_strings():
    for s in range(6):
        assert B.status_string(s).startswith("MOE_")
    assert "unknown" in B.status_string(42)


def test_sharded_entry_points_validate_on_the_host():
    L = B.lib()
    cfg = B.make_config(100, 128, 8, 128, 2, capacity_factor=1.0)
    n = ctypes.c_size_t(0)
    # T_global below this rank's tokens; too many assignments overall
    assert L.moe_sharded_workspace_size(ctypes.byref(cfg), 99, ctypes.byref(n)) == \
        B.MOE_ERR_INVALID_ARG
    assert L.moe_sharded_workspace_size(ctypes.byref(cfg), 1 << 30, ctypes.byref(n)) == \
        B.MOE_ERR_UNSUPPORTED
    # the capacity of the whole batch may keep more rows on one rank than a
    # batch of this rank's size could: the split-batch scratch is never smaller
    need = B.sharded_workspace_size(cfg, 400)
    assert need >= B.workspace_size(cfg)
    fake = [4096 * (i + 1) for i in range(16)]
    ws = 1 << 20

    def finish(n_ranks, rank, ws_bytes=need, ptrs=fake, ws_ptr=ws):
        return L.moe_sharded_finish(ctypes.byref(cfg), 400, n_ranks, rank, *ptrs[:15], ws_ptr,
                                    ctypes.c_size_t(ws_bytes), None)

    for n_ranks, rank in ((2, 2), (0, 0), (4, -1)):
        assert finish(n_ranks, rank) == B.MOE_ERR_INVALID_ARG
    assert finish(4, 1, ws_bytes=need - 1) == B.MOE_ERR_WORKSPACE
    assert finish(4, 1, ws_ptr=ws + 64) == B.MOE_ERR_WORKSPACE
    no_counts = [None] + fake[1:]
    assert finish(4, 1, ptrs=no_counts) == B.MOE_ERR_INVALID_ARG

    def route(ptrs, ws_bytes=need):
        return L.moe_sharded_route(ctypes.byref(cfg), 400, *ptrs, ws, ctypes.c_size_t(ws_bytes),
                                   None)

    r = fake[:8]
    missing_sums = r[:7] + [None]
    assert route(missing_sums) == B.MOE_ERR_INVALID_ARG
    assert route(r, ws_bytes=need - 1) == B.MOE_ERR_WORKSPACE
    misaligned_x = [4096 + 8] + r[1:]
    assert route(misaligned_x) == B.MOE_ERR_INVALID_ARG


def test_launch_plan():
    plan = lambda name: B.launch_plan(B.config_of(WORKLOADS[name]))
    sw = plan("switch_top1_capacity")
    assert sw["router_fused"] and sw["direct_y"] and not sw["shared_fused"]
    # decode-sized layers run the shared expert's tiles inside the routed launches
    for name in ("qwen2_57b_decode", "dsv3_decode"):
        p = plan(name)
        assert p["shared_fused"] and not p["pair_routed"] and not p["pair_shared"], name
    # large layers: CTA pairs, shared expert in its own launches
    q = plan("qwen2_57b_prefill")
    assert q["pair_shared"] and not q["shared_fused"]
    assert plan("mixtral_prefill")["pair_routed"]
    # 256 experts: pair tiles plus 128-row remainder tiles; 64 experts: pairs only
    # every launch on CTA pairs runs the segments' remainders as swap units
    assert plan("dsv3_prefill")["pair_tails"] and q["pair_tails"]
    assert not plan("mixtral_decode")["pair_tails"]
    assert not plan("mixtral_decode")["pair_routed"]
    with pytest.raises(B.MoeError):
        B.launch_plan(B.make_config(64, 128, 8, 128, 0))


def test_barrier_fault_hook_validates_its_arguments():
    """The bounded-wait test hook accepts one extra arrival and limits from
    1 us to the 2 s default, and rejects anything else (host only)."""
    L = B.lib()
    for extra, lim in ((2, 0), (-1, 0), (1, 500), (1, 3_000_000_000)):
        assert L.moe_debug_barrier_fault(extra, lim) == B.MOE_ERR_INVALID_ARG
    assert L.moe_debug_barrier_fault(1, 1_000_000) == B.MOE_OK
    assert L.moe_debug_barrier_fault(0, 0) == B.MOE_OK


def test_latent_offsets_lie_inside_the_workspace():
    cfg = B.make_config(64, 1024, 64, 2048, 8, gating_mode=2)
    xo, yo = B.latent_offsets(cfg, 4096)
    n = 64 * 1024 * 2
    assert xo % 1024 == 0 and yo >= xo + n and yo + n <= B.latent_workspace_size(cfg, 4096)
    with pytest.raises(B.MoeError):
        B.latent_offsets(cfg, 100)       # d_outer not a multiple of 64 for bf16


def test_debug_bounds_build_exports_the_same_symbols():
    """libmoe_debug_bounds.so (the sources built with MOE_DEBUG_BOUNDS) is a
    drop-in replacement: it exports exactly the entry points of libmoe.so."""
    from mixture_experts_layer_capacity_b300 import build
    dbg = build.build(debug_bounds=True)

    def exported(path):
        out = os.popen(f"nm -D --defined-only {path}").read().split("\n")
        return sorted(l.split()[-1] for l in out if " T " in l)

    assert exported(dbg) == exported(B.LIB_PATH)
    assert set(_declared_symbols()) <= set(exported(dbg))
    tl = build.build(timeline=True)
    assert exported(tl) == exported(B.LIB_PATH)


def test_timeline_is_unsupported_outside_its_build():
    """Only libmoe_timeline.so records the pair GEMMs' unit timeline; the
    normal library refuses both calls before touching the device."""
    L = B.lib()
    assert L.moe_timeline_clear() == B.MOE_ERR_UNSUPPORTED
    buf = np.zeros(8, dtype=np.uint64)
    assert L.moe_timeline_read(buf.ctypes.data, 8) == B.MOE_ERR_UNSUPPORTED
    with pytest.raises(B.MoeError):
        B.timeline_read(8)
    assert B.TIMELINE_WORDS == 98304


def test_timeline_build_validates_before_touching_the_device():
    """libmoe_timeline.so refuses a null buffer or a word count outside
    [0, MOE_TIMELINE_WORDS] before any CUDA call (run in a child process,
    which loads that build instead of libmoe.so)."""
    import subprocess
    import sys
    from mixture_experts_layer_capacity_b300 import build
    lib = build.build(timeline=True)
    child = (
        "import ctypes, sys\n"
        "import numpy as np\n"
        "L = ctypes.CDLL(sys.argv[1])\n"
        "L.moe_timeline_read.argtypes = [ctypes.c_void_p, ctypes.c_int64]\n"
        "buf = np.zeros(8, dtype=np.uint64)\n"
        "print(L.moe_timeline_read(None, 8), L.moe_timeline_read(buf.ctypes.data, -1),\n"
        "      L.moe_timeline_read(buf.ctypes.data, 98305))\n")
    r = subprocess.run([sys.executable, "-c", child, lib], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.split() == [str(B.MOE_ERR_INVALID_ARG)] * 3


def _call_w8a8(cfg, ws, ws_bytes, shared=True):
    """moe_forward_w8a8 with fake (never dereferenced) 16-byte aligned
    pointers; returns the status."""
    vals = [4096 * (i + 1) for i in range(23)]
    if not shared:
        for i in range(12, 18):       # Ws_gate_q ... Ws_down_scale
            vals[i - 3] = None
    args = [ctypes.c_void_p(v) if v else None for v in vals] + [ctypes.c_void_p(ws) if ws else None]
    return B.lib().moe_forward_w8a8(ctypes.byref(cfg), *args, ctypes.c_size_t(ws_bytes), None)


def test_w8a8_workspace_and_validation():
    cfg = B.make_config(64, 512, 8, 256, 2, d_shared=256)
    need = B.w8a8_workspace_size(cfg)
    base = B.workspace_size(cfg)
    R, D, F, T, S = 64 * 2, 512, 256, 64, 256
    # the quantized rows, the fp32 hidden rows and their shared-expert copies
    assert need >= base + R * (D + F + 4 * F + 8) + T * (D + S + 4 * S + 8)
    L = B.lib()
    offs = [ctypes.c_size_t(0) for _ in range(5)]
    assert L.moe_w8a8_offsets(ctypes.byref(cfg), *[ctypes.byref(o) for o in offs]) == B.MOE_OK
    xq, xs, hf, hq, hs = (o.value for o in offs)
    assert base <= xq and xq + R * D <= xs and xs + 4 * R <= hf and hf + 4 * R * F <= hq
    assert hq + R * F <= hs and hs + 4 * R <= need
    assert L.moe_w8a8_offsets(ctypes.byref(cfg), None, *[ctypes.byref(o) for o in offs[1:]]) \
        == B.MOE_ERR_INVALID_ARG
    # the bf16 layer's workspace is too small for the quantized activations
    assert _call_w8a8(cfg, 1 << 20, base) == B.MOE_ERR_WORKSPACE
    assert _call_w8a8(cfg, (1 << 20) + 128, need) == B.MOE_ERR_WORKSPACE
    # fp32 layers, and a shared expert with d_expert < 128, are not supported
    f32 = B.make_config(64, 512, 8, 256, 2, d_shared=256, dtype="fp32")
    assert _call_w8a8(f32, 1 << 20, need) == B.MOE_ERR_UNSUPPORTED
    narrow = B.make_config(64, 512, 8, 64, 2, d_shared=256)
    assert _call_w8a8(narrow, 1 << 20, 1 << 30) == B.MOE_ERR_UNSUPPORTED
    # a missing shared weight when the layer has a shared expert
    assert _call_w8a8(cfg, 1 << 20, need, shared=False) == B.MOE_ERR_INVALID_ARG


def test_w8a8_swap_plan_follows_rows_per_expert():
    # at most 64 rows per expert on average: the weights-as-M-operand kernels
    assert B.launch_plan(B.make_config(64, 7168, 256, 2048, 8))["w8a8_swap"]
    assert B.launch_plan(B.make_config(2048, 7168, 256, 2048, 8))["w8a8_swap"]
    assert not B.launch_plan(B.make_config(2049, 7168, 256, 2048, 8))["w8a8_swap"]
    assert not B.launch_plan(B.make_config(16384, 7168, 256, 2048, 8))["w8a8_swap"]
    assert B.launch_plan(B.make_config(64, 4096, 8, 14336, 2))["w8a8_swap"]
