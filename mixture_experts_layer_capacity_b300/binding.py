"""Thin ctypes binding of libmoe.so (C ABI in include/moe.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  PyTorch provides device memory and the stream.  The library is
loaded on first use; if it is missing, loading raises -- there is no other
implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# MOE_LIBRARY selects another build of the same library, e.g. the one with
# index range checks (libmoe_debug_bounds.so, see build.py)
LIB_PATH = os.environ.get("MOE_LIBRARY") or os.path.join(_PKG, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_DEVICE_STATUS = 5

MOE_DTYPE_BF16 = 0
MOE_DTYPE_FP32 = 1

MOE_DEVICE_OK = 0
MOE_DEVICE_NONFINITE_SCORE = 1
MOE_DEVICE_PIPELINE_TIMEOUT = 2
MOE_DEVICE_LAUNCH_MISMATCH = 3
MOE_DEVICE_SHARD_MISMATCH = 4
MOE_DEVICE_INDEX_OUT_OF_RANGE = 5


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


class MoeConfig(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d_model", ctypes.c_int32),
                ("n_experts", ctypes.c_int32), ("d_expert", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("d_shared", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("gating_mode", ctypes.c_int32),
                ("capacity_factor", ctypes.c_float), ("aux_alpha", ctypes.c_float),
                ("bias_selection_only", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def lib():
    """The loaded library (raises if libmoe.so was not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m mixture_experts_layer_capacity_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, cfgp = ctypes.c_void_p, ctypes.POINTER(MoeConfig)
        L.moe_workspace_size.argtypes = [cfgp, ctypes.POINTER(ctypes.c_size_t)]
        L.moe_workspace_size.restype = ctypes.c_int
        L.moe_capacity.argtypes = [cfgp]
        L.moe_capacity.restype = ctypes.c_int64
        L.moe_launch_plan.argtypes = [cfgp, ctypes.POINTER(ctypes.c_int32)]
        L.moe_launch_plan.restype = ctypes.c_int
        L.moe_forward.argtypes = [cfgp] + [vp] * 18 + [ctypes.c_size_t, vp]
        L.moe_forward.restype = ctypes.c_int
        L.moe_forward_no_alloc.argtypes = [cfgp] + [vp] * 17 + [vp]
        L.moe_forward_no_alloc.restype = ctypes.c_int
        L.moe_latent_workspace_size.argtypes = [cfgp, ctypes.c_int32,
                                                ctypes.POINTER(ctypes.c_size_t)]
        L.moe_latent_workspace_size.restype = ctypes.c_int
        L.moe_latent_offsets.argtypes = [cfgp, ctypes.c_int32, ctypes.POINTER(ctypes.c_size_t),
                                         ctypes.POINTER(ctypes.c_size_t)]
        L.moe_latent_offsets.restype = ctypes.c_int
        L.moe_latent_forward.argtypes = [cfgp, ctypes.c_int32] + [vp] * 20 + [ctypes.c_size_t,
                                                                              vp]
        L.moe_latent_forward.restype = ctypes.c_int
        L.moe_quantize_e4m3_rows.argtypes = [ctypes.c_int64, ctypes.c_int64, vp, vp, vp, vp]
        L.moe_quantize_e4m3_rows.restype = ctypes.c_int
        L.moe_forward_w8.argtypes = [cfgp] + [vp] * 24 + [ctypes.c_size_t, vp]
        L.moe_forward_w8.restype = ctypes.c_int
        L.moe_w8a8_workspace_size.argtypes = [cfgp, ctypes.POINTER(ctypes.c_size_t)]
        L.moe_w8a8_workspace_size.restype = ctypes.c_int
        L.moe_forward_w8a8.argtypes = [cfgp] + [vp] * 24 + [ctypes.c_size_t, vp]
        L.moe_forward_w8a8.restype = ctypes.c_int
        L.moe_w8a8_offsets.argtypes = [cfgp] + [ctypes.POINTER(ctypes.c_size_t)] * 5
        L.moe_w8a8_offsets.restype = ctypes.c_int
        L.moe_sharded_workspace_size.argtypes = [cfgp, ctypes.c_int64,
                                                 ctypes.POINTER(ctypes.c_size_t)]
        L.moe_sharded_workspace_size.restype = ctypes.c_int
        L.moe_sharded_route.argtypes = [cfgp, ctypes.c_int64] + [vp] * 9 + [ctypes.c_size_t, vp]
        L.moe_sharded_route.restype = ctypes.c_int
        L.moe_sharded_finish.argtypes = ([cfgp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32]
                                         + [vp] * 16 + [ctypes.c_size_t, vp])
        L.moe_sharded_finish.restype = ctypes.c_int
        L.moe_read_device_status.argtypes = [cfgp, vp, vp, ctypes.POINTER(ctypes.c_int32)]
        L.moe_read_device_status.restype = ctypes.c_int
        L.moe_debug_barrier_fault.argtypes = [ctypes.c_int32, ctypes.c_uint64]
        L.moe_debug_barrier_fault.restype = ctypes.c_int
        L.moe_set_stage_events.argtypes = [vp, ctypes.c_int]
        L.moe_set_stage_events.restype = ctypes.c_int
        L.moe_timeline_clear.argtypes = []
        L.moe_timeline_clear.restype = ctypes.c_int
        L.moe_timeline_read.argtypes = [vp, ctypes.c_int64]
        L.moe_timeline_read.restype = ctypes.c_int
        L.moe_status_string.argtypes = [ctypes.c_int]
        L.moe_status_string.restype = ctypes.c_char_p
        _lib = L
        return L


def status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def make_config(T, d_model, n_experts, d_expert, top_k, d_shared=0, dtype="bf16",
                gating_mode=0, capacity_factor=0.0, aux_alpha=0.01,
                bias_selection_only=False) -> MoeConfig:
    dt = {"bf16": MOE_DTYPE_BF16, "fp32": MOE_DTYPE_FP32}.get(dtype, dtype)
    return MoeConfig(int(T), int(d_model), int(n_experts), int(d_expert), int(top_k),
                     int(d_shared), int(dt), int(gating_mode), float(capacity_factor),
                     float(aux_alpha), int(bool(bias_selection_only)))


def config_of(w) -> MoeConfig:
    """MoeConfig of a workloads.Workload."""
    return make_config(w.T, w.D, w.E, w.F, w.k, w.S, w.dtype, w.mode, w.gamma, w.alpha,
                       bias_selection_only=getattr(w, "sel_bias", False))


PLAN_FLAGS = {"router_fused": 1, "direct_y": 2, "pair_routed": 4, "pair_shared": 8,
              "shared_fused": 16, "pair_tails": 32, "w8a8_swap": 64}


def launch_plan(cfg: MoeConfig) -> dict:
    """Which kernels moe_forward launches for cfg (moe_launch_plan)."""
    flags = ctypes.c_int32(0)
    st = lib().moe_launch_plan(ctypes.byref(cfg), ctypes.byref(flags))
    if st != MOE_OK:
        raise MoeError(st, "moe_launch_plan")
    return {name: bool(flags.value & bit) for name, bit in PLAN_FLAGS.items()}


def router_is_fused(cfg: MoeConfig) -> bool:
    """Whether moe_forward computes the router scores inside its gating kernel."""
    return launch_plan(cfg)["router_fused"]


def direct_y(cfg: MoeConfig) -> bool:
    """Whether the down projection writes y itself (no combine kernel)."""
    return launch_plan(cfg)["direct_y"]


def workspace_size(cfg: MoeConfig) -> int:
    n = ctypes.c_size_t(0)
    st = lib().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n))
    if st != MOE_OK:
        raise MoeError(st, "moe_workspace_size")
    return int(n.value)


def capacity(cfg: MoeConfig) -> int:
    return int(lib().moe_capacity(ctypes.byref(cfg)))


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if isinstance(a, torch.Tensor):
        if not a.is_contiguous():
            raise ValueError("tensors passed to libmoe must be contiguous")
        return a.data_ptr()
    raise TypeError(f"unsupported argument type {type(a)}")


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def moe_forward(cfg: MoeConfig, x, W_r, router_bias, W_gate, W_up, W_down,
                Ws_gate, Ws_up, Ws_down, y, router_logits, topk_idx, topk_w,
                dropped_mask, expert_counts, kept_counts, aux_loss, workspace,
                workspace_bytes=None, stream=None) -> None:
    """Same arguments as the C function; tensors or raw device pointers.
    Raises MoeError on a non-OK status."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    args = [x, W_r, router_bias, W_gate, W_up, W_down, Ws_gate, Ws_up, Ws_down, y,
            router_logits, topk_idx, topk_w, dropped_mask, expert_counts, kept_counts,
            aux_loss, workspace]
    st = lib().moe_forward(ctypes.byref(cfg), *[_ptr(a) for a in args],
                           ctypes.c_size_t(int(workspace_bytes)), _stream(stream))
    if st != MOE_OK:
        raise MoeError(st, "moe_forward")


STATIC_SCRATCH_BYTES = 64 * 1024 * 1024


def moe_forward_no_alloc(cfg: MoeConfig, x, W_r, router_bias, W_gate, W_up, W_down,
                         Ws_gate, Ws_up, Ws_down, y, router_logits, topk_idx, topk_w,
                         dropped_mask, expert_counts, kept_counts, aux_loss,
                         stream=None) -> None:
    """moe_forward without a workspace argument: the library uses its own
    static device scratch (for callers that cannot allocate device memory).
    Raises MoeError on a non-OK status (MOE_ERR_WORKSPACE when the layer
    needs more than STATIC_SCRATCH_BYTES of scratch)."""
    args = [x, W_r, router_bias, W_gate, W_up, W_down, Ws_gate, Ws_up, Ws_down, y,
            router_logits, topk_idx, topk_w, dropped_mask, expert_counts, kept_counts,
            aux_loss]
    st = lib().moe_forward_no_alloc(ctypes.byref(cfg), *[_ptr(a) for a in args],
                                    _stream(stream))
    if st != MOE_OK:
        raise MoeError(st, "moe_forward_no_alloc")


W8_KEYS = ("W_gate", "W_up", "W_down", "Ws_gate", "Ws_up", "Ws_down")


def quantize_e4m3_rows(W: torch.Tensor, stream=None):
    """Row-wise E4M3 codes and fp32 scales of a bf16 device tensor whose last
    dimension is the row (moe_quantize_e4m3_rows): returns (q uint8 of W's
    shape, scale fp32 of W's shape without the last dimension)."""
    if W.dtype != torch.bfloat16 or not W.is_contiguous():
        raise ValueError("quantize_e4m3_rows wants a contiguous bf16 tensor")
    cols = int(W.shape[-1])
    rows = W.numel() // cols
    q = torch.empty(W.shape, dtype=torch.uint8, device=W.device)
    s = torch.empty(W.shape[:-1], dtype=torch.float32, device=W.device)
    st = lib().moe_quantize_e4m3_rows(rows, cols, _ptr(W), _ptr(q), _ptr(s), _stream(stream))
    if st != MOE_OK:
        raise MoeError(st, "moe_quantize_e4m3_rows")
    return q, s


def quantize_expert_weights(inputs: dict, stream=None, a8: bool = False) -> dict:
    """A copy of `inputs` whose expert weights (routed and shared) are E4M3:
    keys W_gate_q / W_gate_s, ... replace W_gate, ...  a8: the layer runs
    with E4M3 activations too (forward calls moe_forward_w8a8)."""
    out = {k: v for k, v in inputs.items() if k not in W8_KEYS}
    for k in W8_KEYS:
        W = inputs.get(k)
        q, s = (None, None) if W is None else quantize_e4m3_rows(W, stream)
        out[k + "_q"], out[k + "_s"] = q, s
    out["a8"] = bool(a8)
    return out


def moe_forward_w8(cfg: MoeConfig, x, W_r, router_bias, W_gate_q, W_gate_s, W_up_q, W_up_s,
                   W_down_q, W_down_s, Ws_gate_q, Ws_gate_s, Ws_up_q, Ws_up_s, Ws_down_q,
                   Ws_down_s, y, router_logits, topk_idx, topk_w, dropped_mask, expert_counts,
                   kept_counts, aux_loss, workspace, workspace_bytes=None, stream=None) -> None:
    """Same arguments as the C function."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    args = [x, W_r, router_bias, W_gate_q, W_gate_s, W_up_q, W_up_s, W_down_q, W_down_s,
            Ws_gate_q, Ws_gate_s, Ws_up_q, Ws_up_s, Ws_down_q, Ws_down_s, y, router_logits,
            topk_idx, topk_w, dropped_mask, expert_counts, kept_counts, aux_loss, workspace]
    st = lib().moe_forward_w8(ctypes.byref(cfg), *[_ptr(a) for a in args],
                              ctypes.c_size_t(int(workspace_bytes)), _stream(stream))
    if st != MOE_OK:
        raise MoeError(st, "moe_forward_w8")


def w8a8_workspace_size(cfg: MoeConfig) -> int:
    n = ctypes.c_size_t(0)
    st = lib().moe_w8a8_workspace_size(ctypes.byref(cfg), ctypes.byref(n))
    if st != MOE_OK:
        raise MoeError(st, "moe_w8a8_workspace_size")
    return int(n.value)


def moe_forward_w8a8(cfg: MoeConfig, x, W_r, router_bias, W_gate_q, W_gate_s, W_up_q, W_up_s,
                     W_down_q, W_down_s, Ws_gate_q, Ws_gate_s, Ws_up_q, Ws_up_s, Ws_down_q,
                     Ws_down_s, y, router_logits, topk_idx, topk_w, dropped_mask, expert_counts,
                     kept_counts, aux_loss, workspace, workspace_bytes=None, stream=None) -> None:
    """Same arguments as the C function."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    args = [x, W_r, router_bias, W_gate_q, W_gate_s, W_up_q, W_up_s, W_down_q, W_down_s,
            Ws_gate_q, Ws_gate_s, Ws_up_q, Ws_up_s, Ws_down_q, Ws_down_s, y, router_logits,
            topk_idx, topk_w, dropped_mask, expert_counts, kept_counts, aux_loss, workspace]
    st = lib().moe_forward_w8a8(ctypes.byref(cfg), *[_ptr(a) for a in args],
                                ctypes.c_size_t(int(workspace_bytes)), _stream(stream))
    if st != MOE_OK:
        raise MoeError(st, "moe_forward_w8a8")


def w8a8_activations(cfg: MoeConfig, workspace: torch.Tensor, rows: int) -> dict:
    """Views of moe_forward_w8a8's quantized activations in `workspace`
    (moe_w8a8_offsets) over the call's first `rows` rows (rows =
    sum(kept_counts)): x_codes uint8 [rows, d_model], x_scales fp32 [rows],
    h_values fp32 [rows, d_expert], h_codes uint8 [rows, d_expert], h_scales
    fp32 [rows]."""
    offs = [ctypes.c_size_t(0) for _ in range(5)]
    st = lib().moe_w8a8_offsets(ctypes.byref(cfg), *[ctypes.byref(o) for o in offs])
    if st != MOE_OK:
        raise MoeError(st, "moe_w8a8_offsets")
    if not 0 <= rows <= cfg.T * cfg.top_k:
        raise ValueError("rows out of range")
    D, F = cfg.d_model, cfg.d_expert
    specs = [("x_codes", torch.uint8, (rows, D), 1), ("x_scales", torch.float32, (rows,), 4),
             ("h_values", torch.float32, (rows, F), 4), ("h_codes", torch.uint8, (rows, F), 1),
             ("h_scales", torch.float32, (rows,), 4)]
    out = {}
    for (name, dt, shape, size), o in zip(specs, offs):
        n = size
        for d in shape:
            n *= d
        out[name] = workspace[o.value:o.value + n].view(dt).view(shape)
    return out


def latent_workspace_size(cfg: MoeConfig, d_outer: int) -> int:
    n = ctypes.c_size_t(0)
    st = lib().moe_latent_workspace_size(ctypes.byref(cfg), int(d_outer), ctypes.byref(n))
    if st != MOE_OK:
        raise MoeError(st, "moe_latent_workspace_size")
    return int(n.value)


def latent_offsets(cfg: MoeConfig, d_outer: int):
    """(x_lat, y_lat) byte offsets of the latent activations inside the
    workspace of moe_latent_forward (moe_latent_offsets)."""
    xo, yo = ctypes.c_size_t(0), ctypes.c_size_t(0)
    st = lib().moe_latent_offsets(ctypes.byref(cfg), int(d_outer), ctypes.byref(xo),
                                  ctypes.byref(yo))
    if st != MOE_OK:
        raise MoeError(st, "moe_latent_offsets")
    return int(xo.value), int(yo.value)


def latent_activations(cfg: MoeConfig, d_outer: int, workspace: torch.Tensor):
    """Views of x_lat and y_lat [T, L] inside a moe_latent_forward workspace."""
    xo, yo = latent_offsets(cfg, d_outer)
    dt = torch.bfloat16 if cfg.dtype == MOE_DTYPE_BF16 else torch.float32
    n = int(cfg.T) * int(cfg.d_model) * (2 if dt == torch.bfloat16 else 4)
    shape = (int(cfg.T), int(cfg.d_model))
    return (workspace[xo:xo + n].view(dt).view(shape),
            workspace[yo:yo + n].view(dt).view(shape))


def moe_latent_forward(cfg: MoeConfig, d_outer, x, W_in, W_out, W_r, router_bias, W_gate,
                       W_up, W_down, Ws_gate, Ws_up, Ws_down, y, router_logits, topk_idx,
                       topk_w, dropped_mask, expert_counts, kept_counts, aux_loss, workspace,
                       workspace_bytes=None, stream=None) -> None:
    """Same arguments as the C function (cfg at the latent width)."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    args = [x, W_in, W_out, W_r, router_bias, W_gate, W_up, W_down, Ws_gate, Ws_up, Ws_down, y,
            router_logits, topk_idx, topk_w, dropped_mask, expert_counts, kept_counts,
            aux_loss, workspace]
    st = lib().moe_latent_forward(ctypes.byref(cfg), int(d_outer), *[_ptr(a) for a in args],
                                  ctypes.c_size_t(int(workspace_bytes)), _stream(stream))
    if st != MOE_OK:
        raise MoeError(st, "moe_latent_forward")


def sharded_workspace_size(cfg: MoeConfig, T_global: int) -> int:
    n = ctypes.c_size_t(0)
    st = lib().moe_sharded_workspace_size(ctypes.byref(cfg), int(T_global), ctypes.byref(n))
    if st != MOE_OK:
        raise MoeError(st, "moe_sharded_workspace_size")
    return int(n.value)


def moe_sharded_route(cfg: MoeConfig, T_global, x, W_r, router_bias, router_logits, topk_idx,
                      topk_w, expert_counts, prob_sums, workspace, workspace_bytes=None,
                      stream=None) -> None:
    """Same arguments as the C function (cfg.T = this rank's tokens)."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    args = [x, W_r, router_bias, router_logits, topk_idx, topk_w, expert_counts, prob_sums,
            workspace]
    st = lib().moe_sharded_route(ctypes.byref(cfg), int(T_global), *[_ptr(a) for a in args],
                                 ctypes.c_size_t(int(workspace_bytes)), _stream(stream))
    if st != MOE_OK:
        raise MoeError(st, "moe_sharded_route")


def moe_sharded_finish(cfg: MoeConfig, T_global, n_ranks, rank, all_expert_counts,
                       all_prob_sums, x, W_gate, W_up, W_down, Ws_gate, Ws_up, Ws_down,
                       topk_idx, topk_w, y, dropped_mask, kept_counts, aux_loss, workspace,
                       workspace_bytes=None, stream=None) -> None:
    """Same arguments as the C function."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    args = [all_expert_counts, all_prob_sums, x, W_gate, W_up, W_down, Ws_gate, Ws_up, Ws_down,
            topk_idx, topk_w, y, dropped_mask, kept_counts, aux_loss, workspace]
    st = lib().moe_sharded_finish(ctypes.byref(cfg), int(T_global), int(n_ranks), int(rank),
                                  *[_ptr(a) for a in args], ctypes.c_size_t(int(workspace_bytes)),
                                  _stream(stream))
    if st != MOE_OK:
        raise MoeError(st, "moe_sharded_finish")


def read_device_status(cfg: MoeConfig, workspace, stream=None) -> int:
    """Synchronises the stream and returns the device status code."""
    code = ctypes.c_int32(0)
    st = lib().moe_read_device_status(ctypes.byref(cfg), _ptr(workspace), _stream(stream),
                                      ctypes.byref(code))
    if st not in (MOE_OK, MOE_ERR_DEVICE_STATUS):
        raise MoeError(st, "moe_read_device_status")
    return int(code.value)


def debug_barrier_fault(extra_arrivals: int, limit_ns: int) -> None:
    """Test hook (moe_debug_barrier_fault): make the routing kernel's grid
    barrier wait for `extra_arrivals` blocks more than exist, giving up after
    limit_ns; (0, 0) restores normal operation."""
    st = lib().moe_debug_barrier_fault(int(extra_arrivals), int(limit_ns))
    if st != MOE_OK:
        raise MoeError(st, "moe_debug_barrier_fault")


NUM_STAGE_EVENTS = 8
STAGES = ("router", "dispatch", "gemm1_routed", "gemm2_routed", "gemm1_shared",
          "gemm2_shared", "combine")


class StageEvents:
    """CUDA events moe_forward records at its stage boundaries (see
    moe_set_stage_events).  Use as a context manager around the calls to
    time; ``elapsed_ms()`` then gives the device time of each stage of the
    last call."""

    def __init__(self):
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(NUM_STAGE_EVENTS)]
        for e in self.events:       # torch creates the CUDA event on first record
            e.record()
        torch.cuda.synchronize()
        self._arr = (ctypes.c_void_p * NUM_STAGE_EVENTS)(*[e.cuda_event for e in self.events])

    def __enter__(self):
        st = lib().moe_set_stage_events(ctypes.cast(self._arr, ctypes.c_void_p),
                                        NUM_STAGE_EVENTS)
        if st != MOE_OK:
            raise MoeError(st, "moe_set_stage_events")
        return self

    def __exit__(self, *exc):
        lib().moe_set_stage_events(None, 0)
        return False

    def elapsed_ms(self) -> dict:
        ev = self.events
        return {name: ev[i].elapsed_time(ev[i + 1]) for i, name in enumerate(STAGES)}


# ---------------------------------------------------------------- convenience
TIMELINE_WORDS = 98304


def timeline_clear() -> None:
    """Zero the per-unit timeline of the routed pair GEMMs (only the library
    built with MOE_TIMELINE has one; others raise MOE_ERR_UNSUPPORTED)."""
    st = lib().moe_timeline_clear()
    if st != MOE_OK:
        raise MoeError(st, "moe_timeline_clear")


def timeline_read(n_words: int = TIMELINE_WORDS):
    """The first n_words of the timeline as a numpy uint64 array (8 words per
    unit: MMA and epilogue phase stamps, see include/moe.h)."""
    import numpy as np
    buf = np.zeros(n_words, dtype=np.uint64)
    st = lib().moe_timeline_read(buf.ctypes.data, n_words)
    if st != MOE_OK:
        raise MoeError(st, "moe_timeline_read")
    return buf


def alloc_outputs(cfg: MoeConfig, device="cuda", d_outer: int = 0, a8: bool = False):
    """Output tensors and workspace for one call, allocated with torch
    (d_outer > 0: for moe_latent_forward, y at the outer width; a8: for
    moe_forward_w8a8)."""
    T, D, E, k = cfg.T, (d_outer or cfg.d_model), cfg.n_experts, cfg.top_k
    dt = torch.bfloat16 if cfg.dtype == MOE_DTYPE_BF16 else torch.float32
    ws_bytes = (latent_workspace_size(cfg, d_outer) if d_outer
                else w8a8_workspace_size(cfg) if a8 else workspace_size(cfg))
    return dict(
        y=torch.empty((T, D), dtype=dt, device=device),
        router_logits=torch.empty((T, E), dtype=torch.float32, device=device),
        topk_idx=torch.empty((T, k), dtype=torch.int32, device=device),
        topk_w=torch.empty((T, k), dtype=torch.float32, device=device),
        dropped_mask=torch.empty((T, k), dtype=torch.uint8, device=device),
        expert_counts=torch.empty((E,), dtype=torch.int32, device=device),
        kept_counts=torch.empty((E,), dtype=torch.int32, device=device),
        aux_loss=torch.empty((1,), dtype=torch.float32, device=device),
        workspace=torch.empty((max(ws_bytes, 256),), dtype=torch.uint8, device=device),
    )


def forward(cfg: MoeConfig, inputs: dict, outs: dict | None = None, stream=None) -> dict:
    """Runs the layer on `inputs` (keys as workloads.make_inputs returns) and
    returns the output dict (allocated if not given).  Inputs with W_in and
    W_out run the latent layer (moe_latent_forward); inputs with E4M3 expert
    weights (quantize_expert_weights) run moe_forward_w8, or moe_forward_w8a8
    when they were quantized with a8."""
    d_outer = int(inputs["x"].shape[1]) if inputs.get("W_in") is not None else 0
    a8 = bool(inputs.get("a8"))
    if outs is None:
        outs = alloc_outputs(cfg, inputs["x"].device, d_outer, a8)
    if inputs.get("W_gate_q") is not None:
        fn = moe_forward_w8a8 if a8 else moe_forward_w8
        fn(cfg, inputs["x"], inputs["W_r"], inputs.get("b_r"),
           *[inputs.get(k + sfx) for k in W8_KEYS for sfx in ("_q", "_s")],
           outs["y"], outs["router_logits"], outs["topk_idx"], outs["topk_w"],
           outs["dropped_mask"], outs["expert_counts"], outs["kept_counts"],
           outs["aux_loss"], outs["workspace"], stream=stream)
        return outs
    if d_outer:
        moe_latent_forward(cfg, d_outer, inputs["x"], inputs["W_in"], inputs["W_out"],
                           inputs["W_r"], inputs.get("b_r"), inputs["W_gate"], inputs["W_up"],
                           inputs["W_down"], inputs.get("Ws_gate"), inputs.get("Ws_up"),
                           inputs.get("Ws_down"), outs["y"], outs["router_logits"],
                           outs["topk_idx"], outs["topk_w"], outs["dropped_mask"],
                           outs["expert_counts"], outs["kept_counts"], outs["aux_loss"],
                           outs["workspace"], stream=stream)
        return outs
    moe_forward(cfg, inputs["x"], inputs["W_r"], inputs.get("b_r"), inputs["W_gate"],
                inputs["W_up"], inputs["W_down"], inputs.get("Ws_gate"), inputs.get("Ws_up"),
                inputs.get("Ws_down"), outs["y"], outs["router_logits"], outs["topk_idx"],
                outs["topk_w"], outs["dropped_mask"], outs["expert_counts"],
                outs["kept_counts"], outs["aux_loss"], outs["workspace"], stream=stream)
    return outs
