"""The attention boundary before the block (providers page,
AttentionBoundaryProvider docstring) on the GPU against the oracle, through
the C ABI: stream (fp32) within 1e-5 of max |stream|, out (bf16) equal after
the near-tie rule (a value within the rounding band of a bf16 midpoint may
land on either neighbour)."""
import numpy as np
import pytest
import torch

import moe_decode_layer_router_gb300 as mm
import oracle as O
import synth
from tests import _harness as H

STREAM_TOL = 1e-5


def _run(name, rows, hidden, eps=1e-6):
    cfg = synth.CONFIGS[name]
    a = synth.attention_boundary_inputs(cfg, rows, hidden)
    partial, w, gate = H.to_dev(a["partial"]), H.to_dev(a["w_pre_ffn_norm"]), H.to_dev(a["gate"])
    stream = H.to_dev(a["stream"])
    out = torch.empty((rows, hidden), dtype=torch.int16, device="cuda")
    mm.musemoe_attention_boundary(partial, stream, out, w, gate, rows, hidden, eps)
    torch.cuda.synchronize()
    s_gpu = stream.cpu().numpy().astype(np.float64)
    o_gpu = O.bf16_to_f64(out.cpu().numpy().view(np.uint16))
    ties = {}
    s_ref, o_ref = O.attention_boundary(a["partial"], a["stream"], float(a["gate"][0]),
                                        a["w_pre_ffn_norm"], eps, near=o_gpu, ties=ties)
    return s_gpu, o_gpu, s_ref, o_ref, ties


@pytest.mark.gpu
@pytest.mark.parametrize("name,rows,hidden", [
    ("decode", 8, 5120),   # the decode workload's rows and hidden size
    ("large", 256, 5120),  # the largest batch
    ("tiny", 4, 256),
    ("decode", 1, 8192),   # the largest row the kernel holds
    ("decode", 3, 2052),   # a ragged row: not a multiple of the CTA's 2048-element pass
    ("decode", 2, 4),      # the smallest
])
def test_attention_boundary_parity(name, rows, hidden):
    s_gpu, o_gpu, s_ref, o_ref, ties = _run(name, rows, hidden)
    assert np.abs(s_gpu - s_ref).max() <= STREAM_TOL * max(1.0, np.abs(s_ref).max())
    np.testing.assert_array_equal(o_gpu, o_ref)
    assert ties.get("out", 0) <= max(2, o_ref.size // 1000)


@pytest.mark.gpu
def test_attention_boundary_zero_gate_keeps_the_stream():
    cfg = synth.CONFIGS["decode"]
    a = synth.attention_boundary_inputs(cfg, 8, 5120)
    partial, w = H.to_dev(a["partial"]), H.to_dev(a["w_pre_ffn_norm"])
    gate = torch.zeros(1, dtype=torch.float32, device="cuda")
    stream = H.to_dev(a["stream"])
    out = torch.empty((8, 5120), dtype=torch.int16, device="cuda")
    mm.musemoe_attention_boundary(partial, stream, out, w, gate, 8, 5120, 1e-6)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(stream.cpu().numpy(), a["stream"])


@pytest.mark.gpu
def test_attention_boundary_rejects_bad_arguments():
    t = torch.zeros((2, 8), dtype=torch.int16, device="cuda")
    s = torch.zeros((2, 8), dtype=torch.float32, device="cuda")
    w = torch.zeros(8, dtype=torch.int16, device="cuda")
    g = torch.zeros(1, dtype=torch.float32, device="cuda")
    for args, word in [((t, s, t, w, g, 0, 8, 1e-6), "rows"),
                       ((t, s, t, w, g, 2, 6, 1e-6), "hidden"),
                       ((t, s, t, w, g, 2, 8, -1.0), "eps"),
                       ((t, None, t, w, g, 2, 8, 1e-6), "stream_io")]:
        with pytest.raises(mm.MuseMoEError) as ei:
            mm.musemoe_attention_boundary(*args)
        assert ei.value.status == mm.MUSEMOE_EINVAL and word in str(ei.value)
