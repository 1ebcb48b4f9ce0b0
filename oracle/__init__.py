"""CPU oracle for one mixture-of-experts FFN layer's forward pass.

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
benchmark's CPU-baseline leg are the only callers.  The arithmetic lives in
``moe_oracle.c`` (plain loops, fp64); this module compiles it with gcc and
marshals numpy arrays.  It imports nothing from the CUDA package, and the
CUDA package imports nothing from here.

Every function cites the page passage it follows in the C source.  The
sampled-row helper :func:`moe_rows` combines per-expert outputs with the same
definition as ``oracle_moe_forward`` (y_t = shared + sum of kept, weighted
expert outputs; [M17] 17.2 equation) for layers whose weights do not fit in
host memory as fp32.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

MODE_SOFTMAX_SELECTED = 0
MODE_SOFTMAX_ALL = 1
MODE_SOFTMAX_ALL_RENORM = 2
MODE_SIGMOID_SELECTED = 3

_ERRORS = {-1: "bad argument", -2: "out of host memory", -3: "non-finite router score"}


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc, -O2, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, i32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        vp = ctypes.c_void_p
        lib.oracle_router_logits.argtypes = [i64, i64, i64, vp, vp, vp, vp]
        lib.oracle_router_logits.restype = None
        lib.oracle_route.argtypes = [i64, i64, i64, i32, vp, vp, vp, vp, vp, vp]
        lib.oracle_route.restype = i32
        lib.oracle_capacity.argtypes = [i64, i64, i64, f64]
        lib.oracle_capacity.restype = i64
        lib.oracle_apply_capacity.argtypes = [i64, i64, i64, i64, vp, vp, vp]
        lib.oracle_apply_capacity.restype = None
        lib.oracle_aux_loss.argtypes = [i64, i64, i64, f64, vp, vp]
        lib.oracle_aux_loss.restype = f64
        lib.oracle_swiglu_rows.argtypes = [i64, i64, i64, vp, vp, vp, vp, vp]
        lib.oracle_swiglu_rows.restype = i32
        lib.oracle_moe_forward.argtypes = (
            [i64, i64, i64, i64, i64, i64, i32, f64, f64, i32] + [vp] * 9 + [vp] * 9)
        lib.oracle_moe_forward.restype = i32
        lib.oracle_linear.argtypes = [i64, i64, i64, vp, vp, vp]
        lib.oracle_linear.restype = None
        lib.oracle_latent_forward.argtypes = (
            [i64, i64, i64, i64, i64, i64, i64, i32, f64, f64, i32] + [vp] * 11 + [vp] * 9)
        lib.oracle_latent_forward.restype = i32
        lib.oracle_e4m3_decode.argtypes = [i64, vp, vp]
        lib.oracle_e4m3_decode.restype = None
        lib.oracle_e4m3_encode.argtypes = [i64, vp, vp]
        lib.oracle_e4m3_encode.restype = None
        lib.oracle_quantize_e4m3_rows.argtypes = [i64, i64, vp, vp, vp]
        lib.oracle_quantize_e4m3_rows.restype = None
        lib.oracle_swiglu_rows_q8.argtypes = [i64, i64, i64] + [vp] * 8
        lib.oracle_swiglu_rows_q8.restype = i32
        lib.oracle_swiglu_rows_w8a8.argtypes = [i64, i64, i64] + [vp] * 8
        lib.oracle_swiglu_rows_w8a8.restype = i32
        _lib = lib
        return lib


def set_threads(n: int) -> int:
    """Sets the number of OpenMP threads the oracle's parallel loops use
    (the process's libgomp) and returns the previous maximum."""
    _load()
    gomp = ctypes.CDLL("libgomp.so.1")
    gomp.omp_get_max_threads.restype = ctypes.c_int
    prev = int(gomp.omp_get_max_threads())
    gomp.omp_set_num_threads(ctypes.c_int(int(n)))
    return prev


def _f32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data


def _check(rc):
    if rc != 0:
        raise RuntimeError(f"oracle: {_ERRORS.get(rc, rc)}")


def router_logits(x, W_r, bias=None):
    """Router scores s = x W_r^T (+ bias), float64 [T, E]."""
    x, W_r = _f32(x), _f32(W_r)
    T, D = x.shape
    E = W_r.shape[0]
    b = None if bias is None else _f32(bias)
    s = np.empty((T, E), dtype=np.float64)
    _load().oracle_router_logits(T, D, E, _ptr(x), _ptr(W_r), _ptr(b), _ptr(s))
    return s


def route(s, k, mode, sel_bias=None):
    """Top-k routing of scores s [T, E] -> (idx int32 [T,k], w f64 [T,k],
    P_sum f64 [E], counts int64 [E]).  sel_bias [E]: a bias that only the
    selection sees (key = fp32(s + b))."""
    s = _f64(s)
    T, E = s.shape
    b = None if sel_bias is None else _f32(sel_bias)
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    P_sum = np.empty(E, dtype=np.float64)
    counts = np.empty(E, dtype=np.int64)
    _check(_load().oracle_route(T, E, k, mode, _ptr(s), _ptr(b), _ptr(idx), _ptr(w),
                                _ptr(P_sum), _ptr(counts)))
    return idx, w, P_sum, counts


def capacity(T, k, E, gamma):
    """Expert capacity ceil(gamma*T*k/E); -1 when gamma <= 0 (dropless)."""
    return int(_load().oracle_capacity(T, k, E, float(gamma)))


def apply_capacity(idx, E, C):
    """Token-order capacity truncation -> (dropped uint8 [T,k], kept int64 [E])."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, k = idx.shape
    dropped = np.empty((T, k), dtype=np.uint8)
    kept = np.empty(E, dtype=np.int64)
    _load().oracle_apply_capacity(T, k, E, int(C), _ptr(idx), _ptr(dropped), _ptr(kept))
    return dropped, kept


def aux_loss(T, k, E, alpha, counts, P_sum):
    """alpha * E * sum_e f_e P_e from demand counts and probability sums."""
    counts = np.ascontiguousarray(counts, dtype=np.int64)
    P_sum = _f64(P_sum)
    return float(_load().oracle_aux_loss(T, k, E, float(alpha), _ptr(counts), _ptr(P_sum)))


def swiglu_rows(x_rows, Wg, Wu, Wd):
    """One SwiGLU expert on rows x [n, D] (fp32 or fp64); Wg, Wu [F, D];
    Wd [D, F] -> f64 [n, D]."""
    x_rows, Wg, Wu, Wd = _f64(x_rows), _f32(Wg), _f32(Wu), _f32(Wd)
    n, D = x_rows.shape
    F = Wg.shape[0]
    out = np.empty((n, D), dtype=np.float64)
    _check(_load().oracle_swiglu_rows(n, D, F, _ptr(x_rows), _ptr(Wg), _ptr(Wu),
                                      _ptr(Wd), _ptr(out)))
    return out


def moe_forward(x, W_r, W_gate, W_up, W_down, *, k, mode, gamma=0.0, alpha=0.0,
                bias=None, Ws_gate=None, Ws_up=None, Ws_down=None, s_in=None,
                bias_selection_only=False):
    """The whole layer on the host.  Returns a dict with s, idx, w, dropped,
    counts, kept, aux, y.  s_in routes on given scores instead of the
    oracle's own.  bias_selection_only: the bias shifts only the selection
    keys (the scores and weights exclude it)."""
    x, W_r = _f32(x), _f32(W_r)
    W_gate, W_up, W_down = _f32(W_gate), _f32(W_up), _f32(W_down)
    T, D = x.shape
    E, F, _ = W_gate.shape
    S = 0 if Ws_gate is None else int(np.asarray(Ws_gate).shape[0])
    Wsg = None if S == 0 else _f32(Ws_gate)
    Wsu = None if S == 0 else _f32(Ws_up)
    Wsd = None if S == 0 else _f32(Ws_down)
    b = None if bias is None else _f32(bias)
    sin = None if s_in is None else _f64(s_in)
    out = dict(
        s=np.empty((T, E), np.float64), idx=np.empty((T, k), np.int32),
        w=np.empty((T, k), np.float64), dropped=np.empty((T, k), np.uint8),
        counts=np.empty(E, np.int64), kept=np.empty(E, np.int64),
        aux=np.empty(1, np.float64), y=np.empty((T, D), np.float64))
    _check(_load().oracle_moe_forward(
        T, D, E, F, k, S, mode, float(gamma), float(alpha), int(bool(bias_selection_only)),
        _ptr(x), _ptr(W_r), _ptr(b), _ptr(W_gate), _ptr(W_up), _ptr(W_down),
        _ptr(Wsg), _ptr(Wsu), _ptr(Wsd), _ptr(sin),
        _ptr(out["s"]), _ptr(out["idx"]), _ptr(out["w"]), _ptr(out["dropped"]),
        _ptr(out["counts"]), _ptr(out["kept"]), _ptr(out["aux"]), _ptr(out["y"])))
    out["aux"] = float(out["aux"][0])
    return out


def linear(x, W):
    """Rows x [n, n_in] (fp32 or fp64) times W [n_out, n_in]^T -> f64 [n, n_out]."""
    x, W = _f64(x), _f32(W)
    n, n_in = x.shape
    out = np.empty((n, W.shape[0]), dtype=np.float64)
    _load().oracle_linear(n, n_in, W.shape[0], _ptr(x), _ptr(W), _ptr(out))
    return out


def latent_forward(x, W_in, W_out, W_r, W_gate, W_up, W_down, *, k, mode, gamma=0.0,
                   alpha=0.0, bias=None, Ws_gate=None, Ws_up=None, Ws_down=None, s_in=None,
                   bias_selection_only=False):
    """A latent MoE: x [T, D_outer] -> x W_in^T [T, L] -> the layer at width L
    -> y_lat W_out^T [T, D_outer].  Same outputs as moe_forward (y at D_outer)."""
    x, W_in, W_out, W_r = _f32(x), _f32(W_in), _f32(W_out), _f32(W_r)
    W_gate, W_up, W_down = _f32(W_gate), _f32(W_up), _f32(W_down)
    T, Do = x.shape
    L = W_in.shape[0]
    E, F, _ = W_gate.shape
    S = 0 if Ws_gate is None else int(np.asarray(Ws_gate).shape[0])
    Wsg = None if S == 0 else _f32(Ws_gate)
    Wsu = None if S == 0 else _f32(Ws_up)
    Wsd = None if S == 0 else _f32(Ws_down)
    b = None if bias is None else _f32(bias)
    sin = None if s_in is None else _f64(s_in)
    out = dict(
        s=np.empty((T, E), np.float64), idx=np.empty((T, k), np.int32),
        w=np.empty((T, k), np.float64), dropped=np.empty((T, k), np.uint8),
        counts=np.empty(E, np.int64), kept=np.empty(E, np.int64),
        aux=np.empty(1, np.float64), y=np.empty((T, Do), np.float64))
    _check(_load().oracle_latent_forward(
        T, Do, L, E, F, k, S, mode, float(gamma), float(alpha), int(bool(bias_selection_only)),
        _ptr(x), _ptr(W_in), _ptr(W_out), _ptr(W_r), _ptr(b), _ptr(W_gate), _ptr(W_up),
        _ptr(W_down), _ptr(Wsg), _ptr(Wsu), _ptr(Wsd), _ptr(sin),
        _ptr(out["s"]), _ptr(out["idx"]), _ptr(out["w"]), _ptr(out["dropped"]),
        _ptr(out["counts"]), _ptr(out["kept"]), _ptr(out["aux"]), _ptr(out["y"])))
    out["aux"] = float(out["aux"][0])
    return out


def e4m3_decode(codes):
    """Values (fp64) of E4M3 codes (uint8 array of any shape)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_e4m3_decode(c.size, _ptr(c), _ptr(out))
    return out


def e4m3_encode(values):
    """E4M3 codes of fp32 values: round to nearest even, saturating."""
    v = _f32(values)
    out = np.empty(v.shape, dtype=np.uint8)
    _load().oracle_e4m3_encode(v.size, _ptr(v), _ptr(out))
    return out


def quantize_e4m3_rows(W):
    """Row-wise E4M3 quantization of W [rows, cols] (fp32 values): returns
    (codes uint8 [rows, cols], scales fp32 [rows])."""
    W = _f32(W)
    rows, cols = W.shape
    q = np.empty((rows, cols), dtype=np.uint8)
    s = np.empty(rows, dtype=np.float32)
    _load().oracle_quantize_e4m3_rows(rows, cols, _ptr(W), _ptr(q), _ptr(s))
    return q, s


def swiglu_rows_q8(x_rows, qg, sg, qu, su, qd, sd):
    """swiglu_rows with E4M3 weights: codes qg, qu [F, D], qd [D, F] and row
    scales sg, su [F], sd [D] -> f64 [n, D]."""
    x_rows = _f64(x_rows)
    qg, qu, qd = (np.ascontiguousarray(a, dtype=np.uint8) for a in (qg, qu, qd))
    sg, su, sd = _f32(sg), _f32(su), _f32(sd)
    n, D = x_rows.shape
    F = qg.shape[0]
    out = np.empty((n, D), dtype=np.float64)
    _check(_load().oracle_swiglu_rows_q8(n, D, F, _ptr(x_rows), _ptr(qg), _ptr(sg), _ptr(qu),
                                         _ptr(su), _ptr(qd), _ptr(sd), _ptr(out)))
    return out


def swiglu_rows_w8a8(x_rows, qg, sg, qu, su, qd, sd):
    """swiglu_rows_q8 with E4M3 activations: each token row and each hidden
    row (rounded to fp32) is quantized row-wise before its projection.
    x_rows [n, D] holds fp32-representable values -> f64 [n, D]."""
    x_rows = _f64(x_rows)
    qg, qu, qd = (np.ascontiguousarray(a, dtype=np.uint8) for a in (qg, qu, qd))
    sg, su, sd = _f32(sg), _f32(su), _f32(sd)
    n, D = x_rows.shape
    F = qg.shape[0]
    out = np.empty((n, D), dtype=np.float64)
    _check(_load().oracle_swiglu_rows_w8a8(n, D, F, _ptr(x_rows), _ptr(qg), _ptr(sg),
                                           _ptr(qu), _ptr(su), _ptr(qd), _ptr(sd), _ptr(out)))
    return out


def _expert_rows(x_rows, weights):
    """One expert on rows: weights = (Wg, Wu, Wd) fp32, the six arrays
    (qg, sg, qu, su, qd, sd) of E4M3 weights, or those six and the string
    "a8" (E4M3 activations too)."""
    if len(weights) == 7 and weights[6] == "a8":
        return swiglu_rows_w8a8(x_rows, *weights[:6])
    if len(weights) == 6:
        return swiglu_rows_q8(x_rows, *weights)
    return swiglu_rows(x_rows, *weights)


def moe_rows(x_rows, idx, w, dropped, expert_weights, shared=None):
    """y rows for a sample of tokens, expert by expert.

    x_rows [n, D] (fp32 or fp64): the sampled tokens' inputs; idx/w/dropped [n, k]: their
    routing (taken from a routing of the whole batch);
    expert_weights(e) -> (Wg [F,D], Wu [F,D], Wd [D,F]) as float32, or the six
    E4M3 arrays (qg, sg, qu, su, qd, sd) of swiglu_rows_q8;
    shared: None or a tuple of the same two kinds.
    Same definition as oracle_moe_forward: y = shared + sum_j kept * w * FFN.
    """
    x_rows = _f64(x_rows)
    n, D = x_rows.shape
    idx = np.asarray(idx)
    w = np.asarray(w, dtype=np.float64)
    dropped = np.asarray(dropped)
    y = np.zeros((n, D), dtype=np.float64)
    for e in sorted(set(int(v) for v in idx[dropped == 0].ravel())):
        rows, slots = np.nonzero((idx == e) & (dropped == 0))
        out = _expert_rows(x_rows[rows], expert_weights(e))
        y[rows] += w[rows, slots][:, None] * out
    if shared is not None:
        y += _expert_rows(x_rows, shared)
    return y
