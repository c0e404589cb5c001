"""Online rounding of BF16 expert weights to MXFP4 (page
"vllm.models.muse_spark.amd.muse_moe_runner", _quantize_experts_to_mxfp4) on
the GPU against the oracle, through the C ABI: codes and scales bit-exact."""
import numpy as np
import pytest
import torch

import moe_decode_layer_router_gb300 as mm
import oracle as O
import synth
from tests import _harness as H


def _gpu(w: np.ndarray):
    rows, cols = w.shape
    wd = H.to_dev(w)
    codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty((rows, cols // 32), dtype=torch.uint8, device="cuda")
    mm.musemoe_quantize_mxfp4(wd, codes, scales, rows, cols)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


@pytest.mark.gpu
@pytest.mark.parametrize("rows,cols,std", [(1, 32, 0.02), (3, 96, 1.0), (128, 2048, 0.02),
                                            (37, 1024, 300.0), (64, 5120, 1e-30)])
def test_quantize_mxfp4_bit_exact(rows, cols, std):
    w = synth.bf16_expert_weights(synth.CONFIGS["decode"], (rows, cols), std)
    codes, scales = _gpu(w)
    want_c, want_s = O.quantize_mxfp4(w)
    np.testing.assert_array_equal(scales, want_s)
    np.testing.assert_array_equal(codes, want_c)


@pytest.mark.gpu
def test_quantize_mxfp4_expert_sized_sampled_rows():
    # w13 of 8 experts of the decode workload: [8 * 2I, P] = [16384, 2048];
    # the oracle checks 64 rows spread over it
    rows, cols = 8 * 2 * 1024, 2048
    w = synth.bf16_expert_weights(synth.CONFIGS["decode"], (rows, cols))
    codes, scales = _gpu(w)
    pick = np.linspace(0, rows - 1, 64).astype(int)
    want_c, want_s = O.quantize_mxfp4(w[pick])
    np.testing.assert_array_equal(scales[pick], want_s)
    np.testing.assert_array_equal(codes[pick], want_c)


@pytest.mark.gpu
def test_quantize_mxfp4_edge_blocks():
    rows = []
    ties = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, -0.25, -0.75, -5.0, -7.0]
    rows.append(ties + [0.0] * 20)                      # ties, saturation
    rows.append([0.0] * 32)                             # zero block
    rows.append([-0.0] * 32)                            # negative zeros
    rows.append([2.0 ** -130, -2.0 ** -133] + [0.0] * 30)  # subnormal amax (clamp)
    rows.append([3.3895313892515355e38, -1.0] + [0.0] * 30)  # largest finite bf16
    rows.append([6.0 * 2.0 ** k for k in range(-16, 16)])   # one binade per element
    w = O.f64_to_bf16_bits(np.array(rows, dtype=np.float64))
    w = np.concatenate([w, w[::-1]], axis=1)            # two blocks per row
    codes, scales = _gpu(np.ascontiguousarray(w))
    want_c, want_s = O.quantize_mxfp4(w)
    np.testing.assert_array_equal(scales, want_s)
    np.testing.assert_array_equal(codes, want_c)


@pytest.mark.gpu
def test_quantize_mxfp4_rejects_bad_arguments():
    w = torch.zeros((2, 64), dtype=torch.int16, device="cuda")
    c = torch.zeros((2, 32), dtype=torch.uint8, device="cuda")
    s = torch.zeros((2, 2), dtype=torch.uint8, device="cuda")
    for args, word in [((w, c, s, 0, 64), "rows"), ((w, c, s, 2, 48), "cols"),
                       ((None, c, s, 2, 64), "w_bf16"), ((w, c, None, 2, 64), "scales")]:
        with pytest.raises(mm.MuseMoEError) as ei:
            mm.musemoe_quantize_mxfp4(*args)
        assert ei.value.status == mm.MUSEMOE_EINVAL and word in str(ei.value)
