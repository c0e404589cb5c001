"""Writes routing_hand_cases.json: hand-worked closed forms of the MuseSpark1x
routing rule (page vllm.models.muse_spark.amd.muse_moe_runner, class
MuseSpark1xRouter) and of the warm-up routing case (page
vllm.models.muse_spark.nvidia.specialized_decode.runtime.providers,
RoutedMoE.warm_up). Uses only the math module: no oracle, no CUDA path."""
import json
import math
import os

ln3 = math.log(3.0)


def sig(z):
    return 1 / (1 + math.exp(-z))


def main():
    spread = [[30.0 if e in (0, 2, 4, 6) else -30.0 for e in range(16)],
              [30.0 if e in (8, 10, 12, 14) else -30.0 for e in range(16)]]
    cases = [
        dict(name="sigmoid_bias_flips_selection", logits=[[0.0, ln3]], bias=[0.3, 0.0], top_k=1,
             score="sigmoid", route_scale=2.5, multiplier=None, division_eps=None, ids=[[0]],
             weights=[[2.5]],
             derivation="s = sigmoid([0, ln 3]) = [1/2, 3/4]; selection = s + bias = [0.8, 0.75] "
                        "picks expert 0; its weight uses the UNBIASED score: 2.5 * 0.5 / 0.5"),
        dict(name="sigmoid_no_bias", logits=[[0.0, ln3]], bias=[0.0, 0.0], top_k=1,
             score="sigmoid", route_scale=2.5, multiplier=None, division_eps=None, ids=[[1]],
             weights=[[2.5]],
             derivation="selection = [0.5, 0.75] picks expert 1; weight 2.5 * 0.75 / 0.75"),
        dict(name="sigmoid_top2_biased_order", logits=[[0.0, ln3]], bias=[0.3, 0.0], top_k=2,
             score="sigmoid", route_scale=2.5, multiplier=None, division_eps=None, ids=[[0, 1]],
             weights=[[1.0, 1.5]],
             derivation="ids in descending selection order [0.8, 0.75]; "
                        "weights 2.5 * [0.5, 0.75] / 1.25"),
        dict(name="sigmoid_top2_unbiased_order", logits=[[0.0, ln3]], bias=[0.0, 0.0], top_k=2,
             score="sigmoid", route_scale=2.5, multiplier=None, division_eps=None, ids=[[1, 0]],
             weights=[[1.5, 1.0]],
             derivation="selection [0.5, 0.75]: ids [1, 0]; weights 2.5 * [0.75, 0.5] / 1.25"),
        dict(name="softmax_top1_division_eps", logits=[[0.0, ln3]], bias=[0.0, 0.0], top_k=1,
             score="softmax", route_scale=2.5, multiplier=None, division_eps=1e-6, ids=[[1]],
             weights=[[2.5 * 0.75 / (0.75 + 1e-6)]],
             derivation="softmax([0, ln 3]) = [1/4, 3/4]; weight 2.5 * 0.75 / (0.75 + 1e-6)"),
        dict(name="multiplier_before_sigmoid", logits=[[2.0, 4.0]], bias=[0.0, 0.0], top_k=2,
             score="sigmoid", route_scale=2.5, multiplier=0.5, division_eps=None, ids=[[1, 0]],
             weights=[[2.5 * sig(2) / (sig(1) + sig(2)), 2.5 * sig(1) / (sig(1) + sig(2))]],
             derivation="the multiplier scales the logits before sigmoid: s = sigmoid([1, 2]); "
                        "weights 2.5 * [s1, s0] / (s0 + s1)"),
        dict(name="all_equal_scores_tie_to_lower_id", logits=[[0.7] * 8], bias=[0.0] * 8,
             top_k=3, score="sigmoid", route_scale=2.5, multiplier=None, division_eps=None,
             ids=[[0, 1, 2]], weights=[[2.5 / 3] * 3],
             derivation="every selection score is equal; reading: equal scores go to the lower id "
                        "first; equal scores give weights 2.5/3"),
        dict(name="warm_up_spread_routes", logits=spread, bias=[0.0] * 16, top_k=4,
             score="sigmoid", route_scale=2.5, multiplier=None, division_eps=None,
             ids=[[0, 2, 4, 6], [8, 10, 12, 14]], weights=[[0.625] * 4, [0.625] * 4],
             derivation="the warm-up routing case: logits -30 everywhere and +30 at b*k experts "
                        "spaced E/(b*k) apart (b=2, k=4, E=16: stride 2); sigmoid(30) rounds to "
                        "1.0 in fp32, so each row picks its four +30 experts with weight 2.5/4"),
    ]
    doc = {"source": "routing rule: page vllm.models.muse_spark.amd.muse_moe_runner, class "
                     "MuseSpark1xRouter (docstring and _compute_routing_native); warm-up case: "
                     "page vllm.models.muse_spark.nvidia.specialized_decode.runtime.providers, "
                     "RoutedMoE.warm_up",
           "note": "hand-worked closed forms; weights are exact values before fp32 storage",
           "cases": cases}
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "routing_hand_cases.json")
    with open(path, "w") as f:
        json.dump(doc, f, indent=1)


if __name__ == "__main__":
    main()
