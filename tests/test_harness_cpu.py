"""Self-test of the GPU tests' comparison logic on the CPU: the oracle's own
outputs, shaped like the GPU taps, must pass it, and planted mistakes in
them must fail it."""
import dataclasses

import numpy as np
import pytest

import synth

from . import _harness as H


@pytest.mark.parametrize("quant", [synth.MXFP4, synth.NVFP4, synth.FP8, synth.BF16,
                                   synth.MXFP4_A4, synth.NVFP4_A4])
def test_oracle_outputs_pass_the_comparison(quant):
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], quant=quant, seed=21)
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    ref = H.oracle_block(cfg, x, st, w)
    rep = H.compare(cfg, w, x, st, H.oracle_as_gpu(cfg, ref))
    assert rep["differ"] == 0 and rep["e2e_out"] == 0.0


@pytest.mark.parametrize("tensor", ["h", "act", "y", "moe_out", "out", "weights"])
def test_planted_mistakes_fail_the_comparison(tensor):
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], seed=22)
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    g = H.oracle_as_gpu(cfg, H.oracle_block(cfg, x, st, w))
    g = {k: np.array(v, copy=True) for k, v in g.items()}
    flat = g[tensor].reshape(-1)
    i = int(np.argmax(np.abs(flat)))
    flat[i] = flat[i] * 1.5 + 0.25
    with pytest.raises(AssertionError):
        H.compare(cfg, w, x, st, g)


def test_bf16_output_error_allows_one_step_only():
    # the independent check of a bf16 output forgives one bf16 step per
    # element (a rounding that went the other way) at any magnitude, and no
    # more: two steps at an element of 4x the RMS still fail the 2e-2 bound
    ref = np.concatenate([[4.3125], np.tile([-0.5, 0.25, 1.0, -1.0, 0.75, -1.25, 0.0078125], 20)])
    rms = float(np.sqrt(np.mean(ref ** 2)))
    assert H.bf16_step(4.3125) == 2.0 ** -5 and H.bf16_step(-0.5) == 2.0 ** -8
    assert H.bf16_step(4.0) == 2.0 ** -5 and H.bf16_step(3.984375) == 2.0 ** -6
    one = ref + np.sign(ref) * H.bf16_step(ref)
    assert H.rel_err_bf16(one, ref) == 0.0
    assert H.rel_err(one, ref) > H.OUT_TOL  # what the plain metric would say
    two = ref.copy()
    two[0] += 2 * H.bf16_step(ref[0])
    assert H.rel_err_bf16(two, ref) == pytest.approx(2.0 ** -5 / rms)
    assert H.rel_err_bf16(two, ref) > H.OUT_TOL


@pytest.mark.parametrize("quant", [synth.MXFP4_A4, synth.NVFP4_A4])
def test_w4a4_without_activation_rounding_fails_the_comparison(quant):
    # a forward that skipped the FP4 rounding of the expert inputs (the W4A16
    # result on the same weights) must not pass as W4A4
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], quant=quant, seed=23)
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    w4a16 = dataclasses.replace(cfg, quant=synth.WEIGHT_FORMAT[quant])
    g = H.oracle_as_gpu(cfg, H.oracle_block(w4a16, x, st, w))
    with pytest.raises(AssertionError):
        H.compare(cfg, w, x, st, g)


def test_kernel_layout_restatement_is_a_permutation():
    rng = np.random.default_rng(0)
    plain = rng.integers(0, 256, size=(2, 128, 512), dtype=np.uint8)
    k = H.kernel_layout(plain, 64, True)
    assert k.shape == plain.shape
    assert np.array_equal(np.sort(k.ravel()), np.sort(plain.ravel()))
    # expert 1, row 73 = tile 1, group 1, row 1; chunk 5 = slice 1, chunk 1 of
    # the slice (8 chunks per row, 4 per slice): offset within the expert
    # 64*512 (tile 1) + 64*4*64 (slice 1) + (1*4 + 1)*512 + 1*64
    off = 64 * 512 + 64 * 4 * 64 + (1 * 4 + 1) * 512 + 64
    blk = k[1].reshape(-1)[off:off + 64]
    row = plain[1, 73, 5 * 64:6 * 64]
    assert np.array_equal(np.sort(blk), np.sort(row))
    # chunk byte 8j + 2q + b sits at 16q + 2j + b (q = 1, j = 3, b = 1)
    assert blk[16 * 1 + 2 * 3 + 1] == row[8 * 3 + 2 * 1 + 1]


def test_kernel_layout_ragged_last_slice():
    rng = np.random.default_rng(1)
    plain = rng.integers(0, 256, size=(1, 64, 5 * 4), dtype=np.uint8)  # 5 chunks of 4 bytes
    k = H.kernel_layout(plain, 4, False)
    # row 9 = group 1, row 1; chunk 4 = the ragged slice 1 holding one chunk:
    # 64*4*4 (slice 0) + (1*1 + 0)*8*4 + 1*4
    off = 64 * 4 * 4 + (1 * 1 + 0) * 8 * 4 + 1 * 4
    assert np.array_equal(k.reshape(-1)[off:off + 4], plain[0, 9, 16:20])
    # and chunk 2 of row 9 in the full slice 0: (1*4 + 2)*8*4 + 1*4
    off = (1 * 4 + 2) * 8 * 4 + 1 * 4
    assert np.array_equal(k.reshape(-1)[off:off + 4], plain[0, 9, 8:12])

def test_kernel_layout_fp8_swizzle():
    rng = np.random.default_rng(2)
    plain = rng.integers(0, 256, size=(1, 64, 128), dtype=np.uint8)  # 2 chunks of 64 B
    k = H.kernel_layout(plain, 64, False, swizzle_fp8=True)
    # row 13 = group 1, row 5: unit u of chunk 1 sits at unit u ^ ((5 >> 1) & 3) = u ^ 2
    blk = k.reshape(-1)[(1 * 2 + 1) * 512 + 5 * 64:(1 * 2 + 1) * 512 + 6 * 64]
    for u in range(4):
        us = u ^ 2
        assert np.array_equal(blk[16 * us:16 * us + 16], plain[0, 13, 64 + 16 * u:64 + 16 * u + 16])
    # row 1 of group 0: (1 >> 1) & 3 = 0, units in place
    blk0 = k.reshape(-1)[64:128]
    assert np.array_equal(blk0, plain[0, 1, :64])


def _self_drift(cfg, seed):
    """The oracle against itself: max |change| / RMS of stream and out when one
    element of every input row moves by one bf16 step (the routing kept)."""
    import oracle as O
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    p = synth.routing_params(cfg)
    a = O.block(x, st, w, quant=cfg.quant, norm_eps=cfg.norm_eps, **p)
    rng = np.random.default_rng(100 + seed)
    xp = x.copy()
    xp[np.arange(x.shape[0]), rng.integers(0, x.shape[1], size=x.shape[0])] += 1
    b = O.block(xp, st, w, quant=cfg.quant, norm_eps=cfg.norm_eps, force_ids=a["ids"], **p)
    return max(H.rel_err(b[k], a[k]) for k in ("stream", "out"))


def test_requantized_forms_drift_beyond_the_w4a16_bound():
    # Why FP8 W8A8 and W4A4 are held to FP8_E2E_TOL independently (and
    # strictly stage-wise): their per-row / per-block dynamic requantization
    # turns a one-step change of one input element per row into a change of
    # the oracle's OWN outputs well beyond the 2e-2 block bound, so no
    # computation that rounds at the pages' points can meet 2e-2 against an
    # independent oracle run; the W4A16 form stays inside it. The bound is
    # within a small multiple of the oracle's own drift (decode shapes, 16
    # experts, 16 rows).
    base = dataclasses.replace(synth.CONFIGS["decode"], rows=16, experts=16, seed=41)
    d = {q: _self_drift(dataclasses.replace(base, quant=q), 0)
         for q in (synth.MXFP4, synth.FP8, synth.MXFP4_A4, synth.NVFP4_A4)}
    assert d[synth.MXFP4] <= H.OUT_TOL, d
    for q in (synth.FP8, synth.MXFP4_A4, synth.NVFP4_A4):
        assert d[q] > H.OUT_TOL, (q, d)
    assert H.FP8_E2E_TOL <= 2.5 * d[synth.FP8], d
