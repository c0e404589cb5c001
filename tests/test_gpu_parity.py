"""Parity of the CUDA path (through the C ABI) with the oracle, element by
element on the same seeded inputs: the full block on every single-layer
workload at full size, its intermediates, and the edge cases."""
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


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    mm.library()


def _compare_block(cfg, w, x, st, run=None, pre_norm=True, report=None):
    """Stage-wise parity (the oracle continues through the GPU's near-tie
    decisions, so every stage is checked on the same inputs) and the
    independent end-to-end parity of the block outputs."""
    t, W = H.upload_layer(cfg, w)
    own = run is None
    run = run or H.Run(cfg, pre_norm=pre_norm)
    try:
        g = run.forward(W, x, st)
        assert mm.musemoe_poll_health(run.handle) == mm.MUSEMOE_OK
    finally:
        if own:
            run.close()
    rep = H.compare(cfg, w, x, st, g, pre_norm=pre_norm)
    if report is not None:
        report.update(rep)
    return g, rep


@pytest.mark.parametrize("name", ["tiny", "decode", "verify", "large", "edge_tiny", "edge",
                                  "w4a4_tiny", "w4a4_nv_tiny", "w4a4", "w4a4_nv"])
def test_block_parity_full_size(name, record_property):
    cfg = synth.CONFIGS[name]
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    rep = {}
    _compare_block(cfg, w, x, st, report=rep)
    for k, v in rep.items():
        record_property(k, v)
    print(name, rep)


@pytest.mark.parametrize("quant", [synth.NVFP4, synth.FP8, synth.BF16, synth.MXFP4_A4,
                                   synth.NVFP4_A4])
@pytest.mark.parametrize("score", [synth.SIGMOID, synth.SOFTMAX])
def test_tiny_dims_every_quant_and_score(quant, score):
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], quant=quant, score=score, seed=11)
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    _compare_block(cfg, w, x, st)


@pytest.mark.parametrize("quant", [synth.MXFP4, synth.NVFP4, synth.FP8, synth.BF16,
                                   synth.MXFP4_A4, synth.NVFP4_A4])
def test_ragged_k_slices(quant):
    # P = 640, I = 384: w13 rows of 5 (FP4) / 10 (FP8) 64-byte chunks and w2
    # rows of 3 / 6 chunks, so the last K-slice of a tile is ragged and tiles
    # are split across CTAs
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], pooled=640, inter=384, quant=quant, seed=12)
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    _compare_block(cfg, w, x, st)


@pytest.mark.parametrize("rows", [1, 3, 13])
def test_ragged_rows(rows):
    # rows below the handle's max_rows, including a ragged tail of a token tile
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], rows=16, seed=5)
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    run = H.Run(cfg, max_rows=16)
    try:
        _compare_block(cfg, w, x[:rows].copy(), st[:rows].copy(), run=run)
    finally:
        run.close()


@pytest.mark.parametrize("quant,rows", [(synth.MXFP4, 24), (synth.FP8, 12), (synth.MXFP4_A4, 20),
                                        (synth.NVFP4_A4, 31)])
def test_wide_pooler_token_blocks_every_form(quant, rows):
    # 9..32 rows: the pooler GEMV takes 16- or 32-row token blocks and the
    # pre-expert norm runs as its own launch (8 rows per CTA, a ragged last
    # CTA), before the FP8 or W4A4 rounding of h
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], rows=rows, quant=quant, seed=12)
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    _compare_block(cfg, w, x, st)


@pytest.mark.parametrize("top_k", [1, 16])
def test_top_k_extremes(top_k):
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], top_k=top_k, seed=6)
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    _compare_block(cfg, w, x, st)


def test_no_multiplier_no_eps_no_pre_norm():
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], multiplier=None, division_eps=None, seed=7)
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    _compare_block(cfg, w, x, st, pre_norm=False)


def test_all_equal_scores_go_to_the_lowest_ids():
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], seed=8)
    w = synth.layer_tensors(cfg)
    w["expert_bias"][:] = 0.0
    x, st = synth.activations(cfg)
    x[:] = 0  # zero input: every logit 0, every score sigmoid(0)
    g, _ = _compare_block(cfg, w, x, st)
    assert (g["ids"] == np.arange(cfg.top_k)).all()
    assert np.all(g["moe_out"] == 0)
    np.testing.assert_array_equal(g["stream"], st.astype(np.float64))


def test_large_rows_multiple_token_groups():
    # 64 rows all routed to the same few experts: token groups of 64 routes
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], rows=64, top_k=2, hot_experts=2,
                              hot_bias=5.0, seed=9)
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    _compare_block(cfg, w, x, st)


@pytest.mark.parametrize("quant,rows", [(synth.NVFP4, 256), (synth.FP8, 64), (synth.BF16, 64),
                                        (synth.BF16, 256), (synth.MXFP4_A4, 64)])
def test_wide_token_tiles_every_form(quant, rows):
    # rows above 32 run the expert kernels with four (up to 64 rows) or eight
    # token tiles per warp; hot experts fill groups of 32 / 64 tokens, whose
    # activation rows ride in the stages beside the weights
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], rows=rows, top_k=2, hot_experts=2,
                              hot_bias=5.0, quant=quant, seed=13)
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    _compare_block(cfg, w, x, st)


def test_route_entry_point_matches_oracle():
    cfg = synth.CONFIGS["decode"]
    d = synth.dense_tensors(cfg, 0)
    x, _ = synth.activations(cfg)
    wr, wb = H.to_dev(d["w_router"]), H.to_dev(d["expert_bias"])
    W = mm.make_weights({"w_router": wr, "expert_bias": wb})
    run = H.Run(cfg)
    try:
        ids = torch.empty((cfg.rows, cfg.top_k), dtype=torch.int32, device="cuda")
        wts = torch.empty((cfg.rows, cfg.top_k), dtype=torch.float32, device="cuda")
        mm.musemoe_route(run.handle, W, H.to_dev(x), cfg.rows, ids, wts)
        torch.cuda.synchronize()
    finally:
        run.close()
    r = O.route(O.router_logits(x, d["w_router"]), d["expert_bias"], cfg.top_k, cfg.route_scale,
                cfg.multiplier, cfg.score, cfg.division_eps)
    gi = ids.cpu().numpy()
    H.check_ids(gi, r, cfg.top_k)
    want = O.weights_for_ids(r.scores, gi, cfg.route_scale, cfg.division_eps)
    np.testing.assert_allclose(wts.cpu().numpy(), want, rtol=H.WEIGHT_RTOL, atol=0)


def test_forward_is_deterministic_and_graph_capturable():
    cfg = synth.CONFIGS["decode"]
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    t, W = H.upload_layer(cfg, w)
    run = H.Run(cfg)
    try:
        xd = H.to_dev(x)
        outs = []
        for _ in range(2):
            sd = H.to_dev(st)
            out = torch.empty((cfg.rows, cfg.hidden), dtype=torch.int16, device="cuda")
            mm.musemoe_forward(run.handle, W, xd, sd, out, cfg.rows)
            torch.cuda.synchronize()
            outs.append((sd.clone(), out.clone()))
        assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
        # capture one forward in a CUDA graph and replay it
        sd = H.to_dev(st)
        out = torch.empty((cfg.rows, cfg.hidden), dtype=torch.int16, device="cuda")
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            mm.musemoe_forward(run.handle, W, xd, sd, out, cfg.rows, s)  # warm
        torch.cuda.synchronize()
        sd.copy_(H.to_dev(st))
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            mm.musemoe_forward(run.handle, W, xd, sd, out, cfg.rows, s)
        sd.copy_(H.to_dev(st))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(sd, outs[0][0]) and torch.equal(out, outs[0][1])
    finally:
        run.close()


def test_forward_host_matches_device_forward():
    cfg = synth.CONFIGS["tiny"]
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    t, W = H.upload_layer(cfg, w)
    run = H.Run(cfg)
    try:
        g = run.forward(W, x, st, taps=False)
        xh = torch.from_numpy(x.view(np.int16).copy()).pin_memory()
        sh = torch.from_numpy(st.copy()).pin_memory()
        oh = torch.empty((cfg.rows, cfg.hidden), dtype=torch.int16).pin_memory()
        mm.musemoe_forward_host(run.handle, W, xh, sh, oh, cfg.rows)
    finally:
        run.close()
    np.testing.assert_array_equal(oh.numpy().view(np.uint16), g["out_bits"])
    np.testing.assert_array_equal(sh.numpy().astype(np.float64), g["stream"])


@pytest.mark.parametrize("dims", [(256, 128), (640, 384)])
@pytest.mark.parametrize("quant", [synth.MXFP4, synth.NVFP4, synth.FP8, synth.BF16])
def test_pack_matches_the_documented_layout(quant, dims):
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], quant=quant, pooled=dims[0], inter=dims[1])
    e = synth.expert_tensors(cfg, 0)
    src = {k: H.to_dev(v) for k, v in e.items()}
    dst = {k: torch.empty_like(v) for k, v in src.items()}
    d = H.dims_of(cfg)
    q = H.QUANT[quant]
    mm.musemoe_pack_experts(d, q, src["w13"], src.get("w13_scale"), dst["w13"],
                            dst.get("w13_scale"), src["w2"], src.get("w2_scale"), dst["w2"],
                            dst.get("w2_scale"))
    mm.musemoe_pack_experts(d, q, src["w13"], src.get("w13_scale"), src["w13"],
                            src.get("w13_scale"), src["w2"], src.get("w2_scale"), src["w2"],
                            src.get("w2_scale"))
    torch.cuda.synchronize()
    for k in ("w13", "w13_scale", "w2", "w2_scale"):
        if k in src:
            assert torch.equal(src[k], dst[k]), k   # in place == out of place
    fp4 = quant in (synth.MXFP4, synth.NVFP4)
    sc = 4 if quant == synth.MXFP4 else 8
    for k in ("w13", "w2"):
        want = H.kernel_layout(e[k], 64, fp4, permute_bf16=quant == synth.BF16,
                               swizzle_fp8=quant == synth.FP8)
        got = dst[k].cpu().numpy().view(np.uint8).reshape(want.shape)
        np.testing.assert_array_equal(got, want)
        if quant == synth.BF16:
            continue  # no scales
        if fp4:
            ws = H.kernel_layout(e[k + "_scale"], sc, False)
            np.testing.assert_array_equal(dst[k + "_scale"].cpu().numpy(), ws)
        else:
            np.testing.assert_array_equal(dst[k + "_scale"].cpu().numpy(), e[k + "_scale"])
