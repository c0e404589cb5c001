"""The C ABI's contract on a GPU: validation before launch, status codes,
error texts, and the health word."""
import dataclasses

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


def test_create_refuses_unsupported_dims_with_every_reason():
    cfg = synth.CONFIGS["tiny"]
    d = H.dims_of(cfg)
    d.pooled, d.top_k, d.experts = 200, 301, 300
    with pytest.raises(mm.MuseMoEError) as ei:
        mm.musemoe_create(d, mm.MUSEMOE_MXFP4, H.config_of(cfg))
    assert ei.value.status == mm.MUSEMOE_EUNSUPPORTED
    msg = str(ei.value)
    assert "pooled 200" in msg and "experts 300" in msg and "top_k 301" in msg
    with pytest.raises(mm.MuseMoEError) as ei:
        mm.musemoe_create(H.dims_of(cfg), 7, H.config_of(cfg))
    assert ei.value.status == mm.MUSEMOE_EUNSUPPORTED


def test_forward_validates_before_launch():
    cfg = synth.CONFIGS["tiny"]
    w = synth.layer_tensors(cfg)
    t, W = H.upload_layer(cfg, w)
    run = H.Run(cfg)
    try:
        x = torch.zeros((cfg.rows, cfg.hidden), dtype=torch.int16, device="cuda")
        s = torch.zeros((cfg.rows, cfg.hidden), dtype=torch.float32, device="cuda")
        o = torch.zeros((cfg.rows, cfg.hidden), dtype=torch.int16, device="cuda")
        for rows in (0, cfg.rows + 1):
            with pytest.raises(mm.MuseMoEError) as ei:
                mm.musemoe_forward(run.handle, W, x, s, o, rows)
            assert ei.value.status == mm.MUSEMOE_EINVAL and "rows" in str(ei.value)
        with pytest.raises(mm.MuseMoEError) as ei:
            mm.musemoe_forward(run.handle, W, x.data_ptr() + 2, s, o, cfg.rows)
        assert ei.value.status == mm.MUSEMOE_EINVAL and "aligned" in str(ei.value)
        bad = mm.make_weights({k: v for k, v in t.items() if k != "w_unpool"})
        with pytest.raises(mm.MuseMoEError) as ei:
            mm.musemoe_forward(run.handle, bad, x, s, o, cfg.rows)
        assert "w_unpool is NULL" in str(ei.value)
        # nothing ran: the output buffers are untouched
        torch.cuda.synchronize()
        assert int(o.abs().sum()) == 0 and float(s.abs().sum()) == 0.0
    finally:
        run.close()


def test_health_reports_fp16_operand_overflow_and_clears():
    cfg = synth.CONFIGS["tiny"]
    w = synth.layer_tensors(cfg)
    # an effective pre-norm weight of 2^17 puts |h| far above 65504
    w["w_pre_norm"][:] = np.uint16(0x4800)
    x, st = synth.activations(cfg)
    t, W = H.upload_layer(cfg, w)
    run = H.Run(cfg)
    try:
        run.forward(W, x, st, taps=False)
        assert mm.musemoe_poll_health(run.handle) == mm.MUSEMOE_ERANGE
        assert "fp16" in mm.musemoe_last_error(run.handle)
        assert mm.musemoe_poll_health(run.handle) == mm.MUSEMOE_OK
    finally:
        run.close()


def test_bounded_waits_time_out_into_the_health_word_and_the_context_survives():
    cfg = synth.CONFIGS["tiny"]
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    t, W = H.upload_layer(cfg, w)
    run = H.Run(cfg)
    try:
        mm.musemoe_health_selftest(run.handle)
        assert mm.musemoe_poll_health(run.handle) == mm.MUSEMOE_ETIMEOUT
        assert mm.musemoe_poll_health(run.handle) == mm.MUSEMOE_OK  # cleared by the poll
        # the context is usable: a forward afterwards still matches the oracle
        H.compare(cfg, w, x, st, run.forward(W, x, st))  # asserts the parity bounds
        assert mm.musemoe_poll_health(run.handle) == mm.MUSEMOE_OK
    finally:
        run.close()


def test_timeout_poll_resets_the_split_tile_tickets():
    # the self-test raises the expert kernels' tickets as contributors that
    # arrived after their owner gave up would leave them; the poll that
    # reports the timeout must zero them. K = 2048 makes four K-slices per
    # tile and 48 rows fewer units per CTA than that, so on the tensor-core
    # path most tiles are split across CTAs: a ticket left raised would let
    # an owner add partials that were never written
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], rows=48, pooled=2048, inter=512, top_k=2,
                              seed=61)
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    t, W = H.upload_layer(cfg, w)
    run = H.Run(cfg)
    try:
        mm.musemoe_set_expert_path(run.handle, mm.MUSEMOE_PATH_TCGEN05)
        H.compare(cfg, w, x, st, run.forward(W, x, st))
        mm.musemoe_health_selftest(run.handle)
        assert mm.musemoe_poll_health(run.handle) == mm.MUSEMOE_ETIMEOUT
        H.compare(cfg, w, x, st, run.forward(W, x, st))
        assert mm.musemoe_poll_health(run.handle) == mm.MUSEMOE_OK
    finally:
        run.close()


def test_num_kernels_and_names():
    assert mm.musemoe_num_kernels(mm.MUSEMOE_MXFP4) == 7
    assert mm.musemoe_num_kernels(mm.MUSEMOE_FP8_W8A8) == 8
    names = [mm.musemoe_kernel_name(mm.MUSEMOE_FP8_W8A8, i) for i in range(8)]
    assert names == ["router", "pool", "w13", "act_quant", "w2", "finalize", "unpool",
                     "boundary"]


def test_events_time_every_kernel():
    cfg = dataclasses.replace(synth.CONFIGS["tiny"])
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    t, W = H.upload_layer(cfg, w)
    run = H.Run(cfg)
    try:
        n = mm.musemoe_num_kernels(mm.MUSEMOE_MXFP4)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n)]
        for e in ev:  # torch creates the CUDA event on its first record
            e.record()
        out = torch.empty((cfg.rows, cfg.hidden), dtype=torch.int16, device="cuda")
        mm.musemoe_forward_debug(run.handle, W, H.to_dev(x), H.to_dev(st), out, cfg.rows, None,
                                 mm.make_taps(events=ev))
        torch.cuda.synchronize()
        ms = [ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(n)]
        assert all(m > 0 for m in ms)
    finally:
        run.close()


def test_pack_refuses_special_ue8m0_codes():
    cfg = synth.CONFIGS["tiny"]
    e = synth.expert_tensors(cfg, 0)
    for bad in (0x00, 0xFF):
        t = {k: H.to_dev(v) for k, v in e.items()}
        t["w2_scale"][3, 5, 1] = bad
        before = t["w13"].clone()
        with pytest.raises(mm.MuseMoEError) as ei:
            mm.musemoe_pack_experts(H.dims_of(cfg), mm.MUSEMOE_MXFP4, t["w13"], t["w13_scale"],
                                    t["w13"], t["w13_scale"], t["w2"], t["w2_scale"], t["w2"],
                                    t["w2_scale"])
        assert ei.value.status == mm.MUSEMOE_EUNSUPPORTED and "UE8M0" in str(ei.value)
        torch.cuda.synchronize()
        assert torch.equal(before, t["w13"])  # nothing was re-laid
