"""Parity of the tensor-core (tcgen05) expert kernels with the oracle, through
the C ABI: the path forced on at small, ragged and wide shapes of every form
it serves (MXFP4, NVFP4, FP8 W8A8 and the W4A4 forms), and the two expert
paths against each other on the same inputs at full size. (The full-size
verify and large workloads of test_gpu_parity.py take this path by default:
more than 32 rows.)"""
import dataclasses

import numpy as np
import pytest

import moe_decode_layer_router_gb300 as mm
import synth
from moe_decode_layer_router_gb300 import _build

from . import _harness as H

pytestmark = pytest.mark.gpu

TC_FORMS = [synth.MXFP4, synth.NVFP4, synth.FP8, synth.MXFP4_A4, synth.NVFP4_A4]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    mm.library()


def _run_path(cfg, w, x, st, path, max_rows=None):
    t, W = H.upload_layer(cfg, w)
    run = H.Run(cfg, max_rows=max_rows)
    try:
        mm.musemoe_set_expert_path(run.handle, path)
        g = run.forward(W, x, st)
        assert mm.musemoe_poll_health(run.handle) == mm.MUSEMOE_OK
    finally:
        run.close()
    return g


@pytest.mark.parametrize("quant", TC_FORMS)
@pytest.mark.parametrize("score", [synth.SIGMOID, synth.SOFTMAX])
def test_tc_tiny_every_form(quant, score):
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], quant=quant, score=score, seed=31)
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    g = _run_path(cfg, w, x, st, mm.MUSEMOE_PATH_TCGEN05)
    H.compare(cfg, w, x, st, g)


@pytest.mark.parametrize("quant", TC_FORMS)
def test_tc_ragged_k_slices(quant):
    # P = 640, I = 384: the last K-slice of every tile is ragged (FP4 w13 rows
    # of 5 chunks, w2 of 3; FP8 10 and 6), tiles split across CTAs
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], pooled=640, inter=384, quant=quant, seed=32)
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    g = _run_path(cfg, w, x, st, mm.MUSEMOE_PATH_TCGEN05)
    H.compare(cfg, w, x, st, g)


@pytest.mark.parametrize("quant,rows", [(synth.NVFP4, 64), (synth.NVFP4, 256), (synth.MXFP4, 100),
                                        (synth.FP8, 64), (synth.FP8, 256),
                                        (synth.NVFP4_A4, 64), (synth.MXFP4_A4, 160)])
def test_tc_hot_experts_full_groups(quant, rows):
    # two hot experts take nearly every route: groups of 64 tokens (N = 64),
    # several groups per expert, and a ragged last group (N padded to 16)
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], rows=rows, top_k=2, hot_experts=2,
                              hot_bias=5.0, quant=quant, seed=33)
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    g = _run_path(cfg, w, x, st, mm.MUSEMOE_PATH_AUTO)
    H.compare(cfg, w, x, st, g)


@pytest.mark.parametrize("rows", [33, 47, 64])
def test_tc_ragged_rows_of_a_larger_handle(rows):
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], rows=64, quant=synth.NVFP4, seed=34)
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    g = _run_path(cfg, w, x[:rows].copy(), st[:rows].copy(), mm.MUSEMOE_PATH_AUTO, max_rows=64)
    H.compare(cfg, w, x[:rows].copy(), st[:rows].copy(), g)


@pytest.mark.parametrize("quant", [synth.NVFP4, synth.FP8])
def test_mma_path_still_serves_wide_tiles(quant):
    # the warp-level kernels forced at 64 rows (four token tiles per warp)
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], rows=64, top_k=2, hot_experts=2,
                              hot_bias=5.0, quant=quant, seed=35)
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    g = _run_path(cfg, w, x, st, mm.MUSEMOE_PATH_MMA)
    H.compare(cfg, w, x, st, g)


@pytest.mark.parametrize("name", ["verify", "large"])
def test_both_paths_match_the_oracle_at_full_size(name):
    # same inputs and operands, fp32 accumulation in different orders: both
    # paths meet the stage-wise and end-to-end bounds on the same inputs and
    # route identically (their route outputs differ where a bf16 rounding of
    # the activation is a near tie, which the stage-wise check resolves)
    cfg = synth.CONFIGS[name]
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    a = _run_path(cfg, w, x, st, mm.MUSEMOE_PATH_TCGEN05)
    b = _run_path(cfg, w, x, st, mm.MUSEMOE_PATH_MMA)
    np.testing.assert_array_equal(a["ids"], b["ids"])
    ra = H.compare(cfg, w, x, st, a)
    rb = H.compare(cfg, w, x, st, b)
    print(name, "tcgen05", ra, "mma", rb)


@pytest.mark.parametrize("quant", [synth.MXFP4_A4, synth.NVFP4_A4])
def test_w4a4_runs_on_the_fp4_tensor_cores_only(quant):
    # the W4A4 weights are packed for the block-scaled FP4 MMA: the
    # warp-level path is refused, AUTO and TCGEN05 accepted
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], quant=quant)
    run = H.Run(cfg)
    try:
        with pytest.raises(mm.MuseMoEError) as ei:
            mm.musemoe_set_expert_path(run.handle, mm.MUSEMOE_PATH_MMA)
        assert ei.value.status == mm.MUSEMOE_EUNSUPPORTED
        mm.musemoe_set_expert_path(run.handle, mm.MUSEMOE_PATH_TCGEN05)
        mm.musemoe_set_expert_path(run.handle, mm.MUSEMOE_PATH_AUTO)
    finally:
        run.close()


def test_tc_path_refused_for_bf16_experts():
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], quant=synth.BF16)
    run = H.Run(cfg)
    try:
        with pytest.raises(mm.MuseMoEError) as ei:
            mm.musemoe_set_expert_path(run.handle, mm.MUSEMOE_PATH_TCGEN05)
        assert ei.value.status == mm.MUSEMOE_EUNSUPPORTED
        with pytest.raises(mm.MuseMoEError) as ei:
            mm.musemoe_set_expert_path(run.handle, 7)
        assert ei.value.status == mm.MUSEMOE_EINVAL
    finally:
        run.close()


@pytest.mark.parametrize("quant,rows", [(synth.MXFP4, 33), (synth.NVFP4, 64), (synth.FP8, 100),
                                        (synth.BF16, 48), (synth.MXFP4_A4, 300)])
def test_dense_tc_front_every_form(quant, rows):
    # above 32 rows the pooler and unpooler run as dense tensor-core GEMMs (two
    # token blocks at 300 rows), the pre-expert norm as its own launch; shapes
    # whose reduction spans many 64-element blocks and tiles split across CTAs
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], rows=rows, hidden=1024, pooled=640,
                              inter=256, quant=quant, seed=36)
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    g = _run_path(cfg, w, x, st, mm.MUSEMOE_PATH_AUTO)
    H.compare(cfg, w, x, st, g)


@pytest.mark.parametrize("rows,hidden", [(40, 1088), (300, 5120)])
def test_dense_tc_cluster_shapes(rows, hidden):
    # the split-K cluster sizes at their edges: 1088 unpooler rows end in a
    # half tile (rows past the end never stored) and split 4 ways; 40 tiles x
    # 2 token blocks are more items than 76, so the unpooler runs one CTA per
    # item, while its pooler splits 8 ways
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], rows=rows, hidden=hidden, pooled=256,
                              inter=128, quant=synth.MXFP4, seed=37)
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    g = _run_path(cfg, w, x, st, mm.MUSEMOE_PATH_AUTO)
    H.compare(cfg, w, x, st, g)
