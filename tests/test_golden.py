"""Values the pages print, checked against the workload definitions used everywhere else."""
import json
import os

from sparse_expert_ffn_softmax_b300.inputs import WORKLOADS

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_mixtral_parameter_count():
    """The Mixtral-shaped workload has the expert matrices the parameter counter assumes."""
    g = json.load(open(os.path.join(GOLDEN, "mixtral_parameters.json")))
    w = WORKLOADS["mixtral_prefill"]
    per_expert = 3 * w.d_model * w.d_ff  # w1 [F,d], w3 [F,d], w2 [d,F]
    total = g["layers"] * w.n_experts * per_expert
    active = g["layers"] * w.top_k * per_expert
    assert round(total / 1e9, 1) == g["total_bn"]
    assert round(active / 1e9, 1) == g["active_bn"]
    assert round(total / active, 1) == g["ratio"]
    assert w.top_k == g["k"]
