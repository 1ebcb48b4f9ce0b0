"""Sizing and roofline arithmetic for one MoE layer (host-side only).

Closed forms from the pages:
  - a SwiGLU expert holds 3*D*F weights (gate, up, down)
    ("Mixture of Experts: More Parameters, Same FLOPs", 'Counting real
    models'; "Mixture of experts" (frontiers track), 'Counting the parameters
    yourself');
  - under uniform routing a batch of B tokens touches E*(1-(1-k/E)^B) of the
    E experts, and an expert that sees t tokens does 2t FLOPs per weight read
    ('Counting real models' and 'What experts cost at serving time');
  - the expert-parallel all-to-all moves k*D*(1 + 2) bytes per token per
    layer with 1-byte dispatch and 2-byte combine (same section; context
    only: expert parallelism is not built here).

The roofline of a forward pass is the slower of its algorithmic FLOPs at the
tensor-core peak and its algorithmic bytes at HBM bandwidth:
  FLOPs = 6*D*F*sum_e kept_e + 6*D*S*T + 2*T*D*E
  bytes = b*(3*D*F*touched + 3*D*S + D*E + 2*T*D)
(touched = experts with at least one kept token; the x_perm/h/z traffic of an
implementation is overhead and is not counted).
"""
from __future__ import annotations


def expert_params(D: int, F: int) -> int:
    return 3 * D * F


def experts_touched(E: int, k: int, B: int) -> float:
    """Expected experts touched by B uniformly routed tokens."""
    return E * (1.0 - (1.0 - k / E) ** B)


def tokens_per_touched_expert(E: int, k: int, B: int) -> float:
    return B * k / experts_touched(E, k, B)


def alltoall_bytes_per_token_layer(k: int, D: int, dispatch_bytes: int = 1,
                                   combine_bytes: int = 2) -> int:
    return k * D * (dispatch_bytes + combine_bytes)


def layer_flops(T: int, D: int, E: int, F: int, S: int, kept_total: int) -> int:
    """Algorithmic FLOPs of one forward pass (router + kept expert rows + shared)."""
    return 6 * D * F * kept_total + 6 * D * S * T + 2 * T * D * E


def layer_bytes(T: int, D: int, E: int, F: int, S: int, touched: int, b: int,
                weight_bytes: int | None = None) -> int:
    """Algorithmic HBM bytes: touched expert weights, shared weights, router, x, y.
    weight_bytes: bytes per expert weight when they are stored narrower than
    the activations (1 for E4M3, plus a 4-byte scale per weight row)."""
    if weight_bytes is None:
        return b * (3 * D * F * touched + 3 * D * S + D * E + 2 * T * D)
    expert = weight_bytes * (3 * D * F * touched + 3 * D * S) + \
        4 * ((2 * F + D) * touched + (2 * S + D if S else 0))
    return expert + b * (D * E + 2 * T * D)


def expert_flops(D: int, F: int, S: int, T: int, kept_total: int) -> int:
    """FLOPs of the grouped SwiGLU GEMMs alone (routed + shared)."""
    return 6 * D * F * kept_total + 6 * D * S * T


def roofline_time_s(flops: float, nbytes: float, tflops: float, gbs: float):
    """(time, bound) with bound 'tensor' or 'hbm'."""
    t_tc = flops / (tflops * 1e12)
    t_hbm = nbytes / (gbs * 1e9)
    return (t_tc, "tensor") if t_tc >= t_hbm else (t_hbm, "hbm")
