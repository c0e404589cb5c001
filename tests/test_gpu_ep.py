"""Expert parallelism through the C ABI on one GPU: musemoe_forward_ep_partial
(a rank's experts only, fp32 partial moe_out) and musemoe_forward_ep_combine
(bf16 of the summed partials, unpooler, FFN boundary). One rank holding every
expert must reproduce musemoe_forward bit for bit; ranks over disjoint expert
ranges, each with only its own experts' weights, must sum to the block the
oracle computes."""
import dataclasses

import numpy as np
import pytest
import torch

import moe_decode_layer_router_gb300 as mm
import oracle as O
import synth
from moe_decode_layer_router_gb300 import _build

from . import _harness as H

pytestmark = pytest.mark.gpu

EXPERT_KEYS = ("w13", "w13_scale", "w13_gscale", "w2", "w2_scale", "w2_gscale")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    mm.library()


def _local_weights(cfg, w, lo, hi):
    """Device weights of a rank holding experts [lo, hi): the expert tensors
    sliced to its experts and packed for hi - lo experts, the rest whole."""
    t = {k: H.to_dev(v) for k, v in w.items() if k not in EXPERT_KEYS}
    for k in EXPERT_KEYS:
        if k in w:
            t[k] = H.to_dev(np.ascontiguousarray(w[k][lo:hi]))
    d = dataclasses.replace(cfg, experts=hi - lo)
    mm.musemoe_pack_experts(H.dims_of(d), H.QUANT[cfg.quant], t["w13"], t.get("w13_scale"),
                            t["w13"], t.get("w13_scale"), t["w2"], t.get("w2_scale"), t["w2"],
                            t.get("w2_scale"))
    torch.cuda.synchronize()
    return t, mm.make_weights(t)


def _ep_run(cfg, w, x, st, ranges, path=mm.MUSEMOE_PATH_AUTO):
    """Every rank's partial on one handle (the ranks run one after another on
    this GPU), summed, then the combine: (stream, out bits, moe_out values)."""
    run = H.Run(cfg)
    try:
        mm.musemoe_set_expert_path(run.handle, path)
        xd = H.to_dev(x)
        total = torch.zeros((cfg.rows, cfg.pooled), dtype=torch.float32, device="cuda")
        keep = []
        for lo, hi in ranges:
            t, W = _local_weights(cfg, w, lo, hi)
            part = torch.empty((cfg.rows, cfg.pooled), dtype=torch.float32, device="cuda")
            mm.musemoe_forward_ep_partial(run.handle, W, xd, part, cfg.rows, lo, hi - lo)
            torch.cuda.synchronize()
            total += part
            keep.append(t)
        tw, W = H.upload_layer(cfg, w)
        sd = H.to_dev(st)
        out = torch.empty((cfg.rows, cfg.hidden), dtype=torch.int16, device="cuda")
        mm.musemoe_forward_ep_combine(run.handle, W, total, sd, out, cfg.rows)
        torch.cuda.synchronize()
        assert mm.musemoe_poll_health(run.handle) == mm.MUSEMOE_OK
    finally:
        run.close()
    return (sd.cpu().numpy().astype(np.float64), out.cpu().numpy().view(np.uint16),
            O.round_bf16(total.cpu().numpy().astype(np.float64)))


@pytest.mark.parametrize("name,path", [("tiny", mm.MUSEMOE_PATH_AUTO),
                                       ("decode", mm.MUSEMOE_PATH_AUTO),
                                       ("verify", mm.MUSEMOE_PATH_TCGEN05)])
def test_one_rank_holding_every_expert_is_the_forward(name, path):
    cfg = synth.CONFIGS[name]
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    s_ep, o_ep, _ = _ep_run(cfg, w, x, st, [(0, cfg.experts)], path)
    t, W = H.upload_layer(cfg, w)
    run = H.Run(cfg)
    try:
        mm.musemoe_set_expert_path(run.handle, path)
        g = run.forward(W, x, st, taps=False)
    finally:
        run.close()
    np.testing.assert_array_equal(o_ep, g["out_bits"])
    np.testing.assert_array_equal(s_ep, g["stream"])


@pytest.mark.parametrize("name,ranks,path", [("tiny", 2, mm.MUSEMOE_PATH_AUTO),
                                             ("decode", 2, mm.MUSEMOE_PATH_AUTO),
                                             ("decode", 4, mm.MUSEMOE_PATH_MMA),
                                             ("verify", 2, mm.MUSEMOE_PATH_AUTO),
                                             ("large", 2, mm.MUSEMOE_PATH_AUTO)])
def test_ranks_sum_to_the_block(name, ranks, path):
    cfg = synth.CONFIGS[name]
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    E = cfg.experts
    ranges = [(r * E // ranks, (r + 1) * E // ranks) for r in range(ranks)]
    s_ep, o_ep, mo_ep = _ep_run(cfg, w, x, st, ranges, path)
    # the summed partials, rounded, are the single-GPU block's moe_out on the
    # same h (the same front): each rank's expert kernels split their work
    # differently, so the fp32 sums (and, at near ties, the bf16 roundings of
    # the SiLU*up activation) differ; within the block bound
    t, W = H.upload_layer(cfg, w)
    run = H.Run(cfg)
    try:
        mm.musemoe_set_expert_path(run.handle, path)
        g = run.forward(W, x, st)
    finally:
        run.close()
    assert H.rel_err(mo_ep, g["moe_out"]) <= H.OUT_TOL
    # and the block's outputs are the oracle's within the block's bounds
    ref = H.oracle_block(cfg, x, st, w)
    bound = H.e2e_bound(cfg)
    assert H.rel_err(s_ep, ref["stream"]) <= bound
    assert H.rel_err(O.bf16_to_f64(o_ep), ref["out"]) <= bound


def test_ep_refuses_bad_ranges():
    cfg = synth.CONFIGS["tiny"]
    w = synth.layer_tensors(cfg)
    x, _ = synth.activations(cfg)
    t, W = H.upload_layer(cfg, w)
    run = H.Run(cfg)
    try:
        part = torch.empty((cfg.rows, cfg.pooled), dtype=torch.float32, device="cuda")
        for lo, n in [(0, 0), (-1, 2), (cfg.experts - 1, 2)]:
            with pytest.raises(mm.MuseMoEError) as ei:
                mm.musemoe_forward_ep_partial(run.handle, W, H.to_dev(x), part, cfg.rows, lo, n)
            assert ei.value.status == mm.MUSEMOE_EINVAL and "expert range" in str(ei.value)
    finally:
        run.close()
