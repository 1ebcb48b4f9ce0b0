"""The roofline/sizing closed forms against the numbers the pages print
('Counting real models' in "Mixture of Experts: More Parameters, Same FLOPs")."""
import json
import os

from conftest import GOLDEN
from mixture_experts_layer_capacity_b300 import roofline as rl


def _g():
    with open(os.path.join(GOLDEN, "moe_arithmetic.json")) as f:
        return json.load(f)


def test_mixtral_sizes():
    m = _g()["mixtral"]
    one = rl.expert_params(m["D"], m["F"])
    assert round(one / 1e6) == m["one_expert_M"]
    assert round(one * m["E"] * m["layers"] / 1e9, 1) == m["all_experts_B"]
    assert round(one * m["k"] * m["layers"] / 1e9, 1) == m["used_per_token_B"]


def test_deepseek_v3_sizes():
    d = _g()["deepseek_v3"]
    moe_layers = d["layers"] - d["dense_layers"]
    one = rl.expert_params(d["D"], d["F"])
    assert round(one / 1e6) == d["one_expert_M"]
    assert round(one * d["E"] * moe_layers / 1e9) == d["routed_all_B"]
    used = one * (d["k"] + d["shared"]) * moe_layers \
        + rl.expert_params(d["D"], d["F_dense"]) * d["dense_layers"]
    assert round(used / 1e9, 1) == d["used_per_token_B"]
    per_layer = rl.alltoall_bytes_per_token_layer(d["k"], d["D"])
    assert round(per_layer / 1024) == d["alltoall_KiB_per_layer"]
    assert round(per_layer * moe_layers / 2 ** 20, 1) == d["alltoall_MiB_all_layers"]


def test_experts_touched_table():
    t = _g()["touched"]
    for B, touched, per in t["rows"]:
        assert round(rl.experts_touched(t["E"], t["k"], B), 1) == touched
        assert round(rl.tokens_per_touched_expert(t["E"], t["k"], B), 1) == per


def test_layer_flops_and_bytes():
    # Mixtral-shaped layer at T=8192, dropless top-2: 16384 kept rows
    f = rl.layer_flops(8192, 4096, 8, 14336, 0, 16384)
    assert abs(f / 1e9 - 5773.0) < 1.0
    b = rl.layer_bytes(64, 4096, 8, 14336, 0, 8, 2)
    assert abs(b / 1e9 - 2.82) < 0.01
    t, bound = rl.roofline_time_s(f, rl.layer_bytes(8192, 4096, 8, 14336, 0, 8, 2),
                                  1637.7, 6444.1)
    assert bound == "tensor" and 3.4e-3 < t < 3.7e-3
