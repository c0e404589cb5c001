"""Stage-wise oracle check of one layer of the 60-layer stack on every row,
run in worker processes (spawned, no GPU): the oracle starts from the GPU's
layer input and continues through the GPU's near-tie decisions; every stage
must match on the same inputs. Returns the layer's stage errors and near-tie
counts."""
from __future__ import annotations

import numpy as np

import oracle as O
import synth

from . import _harness as H


def _layer(cfg, layer: int, ids) -> dict:
    """The layer's weights with only the experts in ``ids`` generated (the
    others stay zero: the oracle, forced to these ids, never reads them)."""
    w = synth.dense_tensors(cfg, layer)
    full = synth.expert_tensors(cfg, layer, 0, 1)
    for k, v in full.items():
        w[k] = np.zeros((cfg.experts,) + v.shape[1:], dtype=v.dtype)
    for e in np.unique(ids):
        for k, v in synth.expert_tensors(cfg, layer, int(e), 1).items():
            w[k][e] = v[0]
    return w


def check_layer(args) -> dict:
    layer, x_bits, stream, g = args
    cfg = synth.CONFIGS["stack"]
    w = _layer(cfg, layer, g["ids"])
    gids = g["ids"]
    H.check_ids(gids, O.route(O.router_logits(x_bits, w["w_router"]), w["expert_bias"],
                              cfg.top_k, cfg.route_scale, cfg.multiplier, cfg.score,
                              cfg.division_eps), cfg.top_k)
    near = dict(h=g["h"], act=np.where(np.abs(g["act"]) >= 2.0 ** -14, g["act"], np.nan),
                moe_out=g["moe_out"], out=g["out"])
    ref = H.oracle_block(cfg, x_bits, stream, w, force_ids=gids, near=near)
    np.testing.assert_allclose(g["weights"], ref["weights"], rtol=H.WEIGHT_RTOL)
    errs = {"h": H.rel_err(g["h"], ref["h"]), "moe_out": H.rel_err(g["moe_out"], ref["moe_out"]),
            "u": H.rel_err(g["u"], ref["u"]), "stream": H.rel_err(g["stream"], ref["stream"]),
            "out": H.rel_err(g["out"], ref["out"])}
    bad = {k: v for k, v in errs.items() if v > H.STAGE_TOL[k]}
    return {"layer": layer, "errs": errs, "bad": bad, "near_ties": ref["near_ties"]}


def run_chains(args) -> dict:
    """The oracle's own chains through all layers on the sample rows:
    ``tracked`` carries its own state and takes the GPU's value only at near
    ties; ``independent`` carries its own state with its own roundings and
    the GPU's expert selection; ``perturbed`` is the independent chain from an
    input one bf16 step away in one element of each row (the independent
    chain's selection). Returns each chain's final stream and out."""
    kind, x0, st0, per_layer = args
    cfg = synth.CONFIGS["stack"]
    if kind == "tracked":
        x, s = x0.copy(), st0.copy()
        for layer, rec in enumerate(per_layer):
            w = _layer(cfg, layer, rec["ids"])
            H.check_ids(rec["ids"], O.route(O.router_logits(x, w["w_router"]), w["expert_bias"],
                                            cfg.top_k, cfg.route_scale, cfg.multiplier, cfg.score,
                                            cfg.division_eps), cfg.top_k)
            near = dict(h=rec["h"], act=np.where(np.abs(rec["act"]) >= 2.0 ** -14, rec["act"],
                                                 np.nan), moe_out=rec["moe_out"], out=rec["out"])
            r = H.oracle_block(cfg, x, s, w, force_ids=rec["ids"], near=near)
            x, s = r["out_bits"], r["stream"]
        return {"tracked": (s, x)}
    xi, si = x0.copy(), st0.copy()
    xp, sp = x0.copy(), st0.copy()
    xp[:, 0] += 1  # one bf16 step
    for layer, rec in enumerate(per_layer):
        w = _layer(cfg, layer, rec["ids"])
        ind = H.oracle_block(cfg, xi, si, w, force_ids=rec["ids"])
        per = H.oracle_block(cfg, xp, sp, w, force_ids=ind["ids"])
        xi, si = ind["out_bits"], ind["stream"]
        xp, sp = per["out_bits"], per["stream"]
    return {"independent": (si, xi), "perturbed": (sp, xp)}
