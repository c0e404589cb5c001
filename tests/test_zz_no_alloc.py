"""musemoe_route_static: the routing entry point for callers that cannot
allocate device memory (their device memory belongs to another allocator,
e.g. a serving engine's pooled one, or they run where a new allocation is not
allowed). It takes no handle and uses the library's fixed static scratch.

Checked through the C ABI against the handle-based musemoe_route on the same
inputs, on two calls in a row (the second reuses the scratch the first left
behind), within the routing tolerances the other tests use. This file is
collected last, and also runs alone in a fresh process."""
import numpy as np
import pytest
import torch

import moe_decode_layer_router_gb300 as mm
import synth
from moe_decode_layer_router_gb300 import _build

from . import _harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    mm.library()


def _route_both(cfg, run, x, d):
    wr, wb, xd = H.to_dev(d["w_router"]), H.to_dev(d["expert_bias"]), H.to_dev(x)
    b, k = x.shape[0], cfg.top_k
    ids_a = torch.empty((b, k), dtype=torch.int32, device="cuda")
    w_a = torch.empty((b, k), dtype=torch.float32, device="cuda")
    ids_b = torch.full((b, k), -1, dtype=torch.int32, device="cuda")
    w_b = torch.zeros((b, k), dtype=torch.float32, device="cuda")
    W = mm.make_weights({"w_router": wr, "expert_bias": wb})
    mm.musemoe_route(run.handle, W, xd, b, ids_a, w_a)
    mm.musemoe_route_static(cfg.hidden, cfg.experts, cfg.top_k, H.config_of(cfg), wr, wb, xd, b,
                            ids_b, w_b)
    torch.cuda.synchronize()
    return ids_a.cpu().numpy(), w_a.cpu().numpy(), ids_b.cpu().numpy(), w_b.cpu().numpy()


@pytest.mark.parametrize("name", ["decode", "verify"])
def test_route_static_matches_route_on_two_calls(name):
    cfg = synth.CONFIGS[name]
    d = synth.dense_tensors(cfg, 0)
    run = H.Run(cfg)
    try:
        for call in range(2):
            c = synth.Config(**{**cfg.__dict__, "seed": cfg.seed + 100 * call})
            x, _ = synth.activations(c)
            ids_a, w_a, ids_b, w_b = _route_both(cfg, run, x, d)
            np.testing.assert_array_equal(ids_b, ids_a)
            np.testing.assert_allclose(w_b, w_a, rtol=H.WEIGHT_RTOL, atol=0)
    finally:
        run.close()


def test_route_static_allocates_nothing():
    # every buffer exists before the measurement and the first call (which
    # loads the library's code and scratch onto the device) is outside it:
    # the device's free memory must not move across the calls that follow
    cfg = synth.CONFIGS["verify"]
    d = synth.dense_tensors(cfg, 0)
    x, _ = synth.activations(cfg)
    wr, wb, xd = H.to_dev(d["w_router"]), H.to_dev(d["expert_bias"]), H.to_dev(x)
    b, k = x.shape[0], cfg.top_k
    ids = torch.empty((b, k), dtype=torch.int32, device="cuda")
    wts = torch.empty((b, k), dtype=torch.float32, device="cuda")
    conf = H.config_of(cfg)

    def call():
        mm.musemoe_route_static(cfg.hidden, cfg.experts, cfg.top_k, conf, wr, wb, xd, b, ids, wts)

    call()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)


def test_route_static_refuses_a_hidden_beyond_the_router_row():
    cfg = synth.CONFIGS["decode"]
    H_ = 8192 + 64
    x = torch.zeros((1, H_), dtype=torch.int16, device="cuda")
    w = torch.zeros((cfg.experts, H_), dtype=torch.float32, device="cuda")
    bias = torch.zeros((cfg.experts,), dtype=torch.float32, device="cuda")
    ids = torch.zeros((1, cfg.top_k), dtype=torch.int32, device="cuda")
    wts = torch.zeros((1, cfg.top_k), dtype=torch.float32, device="cuda")
    with pytest.raises(mm.MuseMoEError) as ei:
        mm.musemoe_route_static(H_, cfg.experts, cfg.top_k, H.config_of(cfg), w, bias, x, 1,
                                ids, wts)
    assert ei.value.status == mm.MUSEMOE_EUNSUPPORTED and "8192" in str(ei.value)


def test_route_static_rejects_rows_beyond_its_scratch():
    cfg = synth.CONFIGS["decode"]
    n = mm.MUSEMOE_STATIC_MAX_ROWS + 1
    x = torch.zeros((n, cfg.hidden), dtype=torch.int16, device="cuda")
    w = torch.zeros((cfg.experts, cfg.hidden), dtype=torch.float32, device="cuda")
    bias = torch.zeros((cfg.experts,), dtype=torch.float32, device="cuda")
    ids = torch.zeros((n, cfg.top_k), dtype=torch.int32, device="cuda")
    wts = torch.zeros((n, cfg.top_k), dtype=torch.float32, device="cuda")
    with pytest.raises(mm.MuseMoEError) as ei:
        mm.musemoe_route_static(cfg.hidden, cfg.experts, cfg.top_k, H.config_of(cfg), w, bias, x,
                                n, ids, wts)
    assert ei.value.status == mm.MUSEMOE_EINVAL and "static scratch" in str(ei.value)
