"""The C oracle (plain single-threaded C, float64) against the numpy oracle:
bit for bit on every stored output, on every expert form and routing
variant, plus the routing hand cases of tests/golden. The OpenMP build of the
same source must agree bit for bit with the single-threaded one (rows and
routes are independent; each sum stays sequential inside one thread)."""
import dataclasses
import json
import os

import numpy as np
import pytest

import synth
from oracle import c_oracle as C
from oracle import musemoe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SMALL = dict(hidden=512, pooled=256, inter=128, experts=16)


def _variants():
    out = []
    for i, q in enumerate(["mxfp4", "nvfp4", "fp8", "bf16", "mxfp4_a4", "nvfp4_a4"]):
        out.append(synth.Config(f"c_{q}", rows=5, top_k=3, quant=q, seed=40 + i, **SMALL))
    base = synth.Config("c_route", rows=7, top_k=4, quant="mxfp4", seed=50, **SMALL)
    out += [dataclasses.replace(base, name="c_softmax_eps", score="softmax", division_eps=1e-6),
            dataclasses.replace(base, name="c_no_mult_no_eps", multiplier=None,
                                division_eps=None),
            dataclasses.replace(base, name="c_mult_hot", multiplier=0.5, hot_experts=4,
                                seed=51),
            dataclasses.replace(base, name="c_one_row_k1", rows=1, top_k=1, seed=52)]
    return out


def _compare(cfg, pre_norm=True, omp=False):
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    p = synth.routing_params(cfg)
    a = O.block(x, st, w, quant=cfg.quant, norm_eps=cfg.norm_eps, pre_norm=pre_norm, **p)
    b = C.block(x, st, w, quant=cfg.quant, norm_eps=cfg.norm_eps, pre_norm=pre_norm, omp=omp,
                **p)
    np.testing.assert_array_equal(b["ids"], a["ids"])
    np.testing.assert_array_equal(b["weights"], a["weights"].astype(np.float32))
    np.testing.assert_array_equal(b["h"], O.f64_to_bf16_bits(a["h"]))
    np.testing.assert_array_equal(b["moe_out"], O.f64_to_bf16_bits(a["moe_out"]))
    np.testing.assert_array_equal(b["stream"], a["stream"].astype(np.float32))
    np.testing.assert_array_equal(b["out"], a["out_bits"])
    return b


@pytest.mark.parametrize("cfg", _variants(), ids=lambda c: c.name)
def test_c_oracle_matches_numpy_oracle_bit_for_bit(cfg):
    _compare(cfg)


def test_c_oracle_without_pre_expert_norm():
    _compare(synth.Config("c_nonorm", rows=3, top_k=2, quant="nvfp4", seed=60, **SMALL),
             pre_norm=False)


def test_c_oracle_full_width_decode_rows():
    """The full model widths (H 5120, P 2048, I 1024, 128 experts, k 8) on two
    rows, so that every loop runs at its real trip count."""
    cfg = dataclasses.replace(synth.CONFIGS["decode"], rows=2)
    _compare(cfg)


@pytest.mark.parametrize("quant", ["mxfp4", "fp8", "nvfp4_a4"])
def test_openmp_build_matches_single_thread(quant):
    cfg = synth.Config(f"c_omp_{quant}", rows=9, top_k=3, quant=quant, seed=70, **SMALL)
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    p = synth.routing_params(cfg)
    one = C.block(x, st, w, quant=quant, norm_eps=cfg.norm_eps, **p)
    many = C.block(x, st, w, quant=quant, norm_eps=cfg.norm_eps, omp=True, **p)
    for k in one:
        np.testing.assert_array_equal(many[k], one[k], err_msg=k)


def test_c_routing_hand_cases():
    with open(os.path.join(GOLDEN, "routing_hand_cases.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        lg = np.array(case["logits"], np.float64).astype(np.float32)
        ids, wts = C.route(lg, np.array(case["bias"], np.float32), case["top_k"],
                           case["route_scale"], case["multiplier"], case["score"],
                           case["division_eps"])
        assert ids.tolist() == case["ids"], case["name"]
        np.testing.assert_allclose(wts, case["weights"], rtol=2e-7, atol=0, err_msg=case["name"])
