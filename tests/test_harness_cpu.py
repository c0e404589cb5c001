"""Self-test of the GPU tests' comparison logic on the CPU: the oracle's own
outputs, shaped like the GPU taps, must pass it, and planted mistakes in
them must fail it."""
import dataclasses

import numpy as np
import pytest

import synth

from . import _harness as H


@pytest.mark.parametrize("quant", [synth.MXFP4, synth.NVFP4, synth.FP8])
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


def test_kernel_layout_restatement_is_a_permutation():
    cfg = synth.CONFIGS["tiny"]
    e = synth.expert_tensors(cfg, 0, e0=0, ne=2)
    k = H.kernel_layout(e["w13"], 64, True)
    assert k.shape == e["w13"].shape
    assert np.array_equal(np.sort(k.ravel()), np.sort(e["w13"].ravel()))
    # row 9 of expert 1 (group 1, row 1), chunk 0: its 64 plain bytes land at
    # [1][1][0][1] of [E][N/8][chunk][8][64] in permuted order
    flat = k.reshape(2, -1)
    nc = e["w13"].shape[2] // 64
    blk = flat[1, (1 * nc + 0) * 512 + 1 * 64:(1 * nc + 0) * 512 + 2 * 64]
    assert np.array_equal(np.sort(blk), np.sort(e["w13"][1, 9, :64]))
    assert blk[16 * 1 + 2 * 3 + 1] == e["w13"][1, 9, 8 * 3 + 2 * 1 + 1]
