"""The NVFP4 expert input of the W4A4 form (page
"vllm.models.muse_spark.nvidia.specialized_decode.runtime.providers",
ExpertsInput: e2m1 codes with one e4m3 block scale per 16) on the GPU
against the oracle, through the C ABI: codes and scales bit-exact."""
import numpy as np
import pytest
import torch

import moe_decode_layer_router_gb300 as mm
import oracle as O
import synth
from tests import _harness as H


def _gpu(x: np.ndarray):
    rows, cols = x.shape
    xd = H.to_dev(x)
    codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty((rows, cols // 16), dtype=torch.uint8, device="cuda")
    mm.musemoe_quantize_act_nvfp4(xd, codes, scales, rows, cols)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


@pytest.mark.gpu
@pytest.mark.parametrize("rows,cols,std", [(1, 16, 1.0), (3, 48, 1.0), (8, 2048, 1.0),
                                            (64, 1024, 0.05), (37, 512, 3000.0),
                                            (16, 256, 1e-4)])
def test_quantize_act_nvfp4_bit_exact(rows, cols, std):
    x = synth.normal_bf16(31, synth.T_X, (rows, cols), 0.0, std)
    codes, scales = _gpu(x)
    want_c, want_s = O.quantize_act_nvfp4(O.bf16_to_f64(x))
    np.testing.assert_array_equal(scales, want_s)
    np.testing.assert_array_equal(codes, want_c)


@pytest.mark.gpu
def test_quantize_act_nvfp4_edge_blocks():
    rows = [
        [6, -3, 1.5, 0.5, 0, 2, -4, 1, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -6],  # midpoints
        [7, 1.125, -0.5625] + [0] * 13,                  # scale rounds down, code saturates
        [0, -0.0] + [0] * 14,                            # scale 0, sign kept
        [2944, 448] + [0] * 14,                          # scale saturates at 448
        [2.0 ** -12, -(2.0 ** -13)] + [0] * 14,          # scale underflows to 0
        [3 * 2.0 ** -8, 2.0 ** -10] + [0] * 14,          # smallest subnormal scale
        [3.3895313892515355e38, -1.0] + [0] * 14,        # largest finite bf16
        [6.0 * 2.0 ** k for k in range(-8, 8)],          # one binade per element
    ]
    x = O.f64_to_bf16_bits(np.array(rows, dtype=np.float64))
    x = np.ascontiguousarray(np.concatenate([x, x[::-1]], axis=1))  # two blocks per row
    codes, scales = _gpu(x)
    want_c, want_s = O.quantize_act_nvfp4(O.bf16_to_f64(x))
    np.testing.assert_array_equal(scales, want_s)
    np.testing.assert_array_equal(codes, want_c)


@pytest.mark.gpu
def test_quantize_act_nvfp4_rejects_bad_arguments():
    x = torch.zeros((2, 64), dtype=torch.int16, device="cuda")
    c = torch.zeros((2, 32), dtype=torch.uint8, device="cuda")
    s = torch.zeros((2, 4), dtype=torch.uint8, device="cuda")
    for args, word in [((x, c, s, 0, 64), "rows"), ((x, c, s, 2, 40), "cols"),
                       ((None, c, s, 2, 64), "x_bf16"), ((x, c, None, 2, 64), "scales")]:
        with pytest.raises(mm.MuseMoEError) as ei:
            mm.musemoe_quantize_act_nvfp4(*args)
        assert ei.value.status == mm.MUSEMOE_EINVAL and word in str(ei.value)
