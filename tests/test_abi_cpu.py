"""The C ABI library builds, loads and exports every entry point the header
declares; without a GPU, create fails cleanly with a status and a reason.
CPU only (no kernel is launched)."""
import ctypes
import os
import re

import pytest

import moe_decode_layer_router_gb300 as mm
from moe_decode_layer_router_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "musemoe.h")


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(musemoe_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return mm.library()


def test_header_and_binding_agree():
    assert _declared() == sorted(mm.EXPORTED_SYMBOLS)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_workspace_bytes_and_names_need_no_gpu(lib):
    d = mm.Dims(max_rows=8, hidden=5120, pooled=2048, inter=1024, experts=128, top_k=8)
    assert mm.musemoe_workspace_bytes(d, mm.MUSEMOE_MXFP4) > 8 * 8 * 2048 * 4  # >= y
    bad = mm.Dims(max_rows=8, hidden=5120, pooled=2000, inter=1024, experts=128, top_k=8)
    assert mm.musemoe_workspace_bytes(bad, mm.MUSEMOE_MXFP4) == 0
    assert mm.musemoe_kernel_name(mm.MUSEMOE_MXFP4, 2) == "w13"
    assert mm.musemoe_num_kernels(mm.MUSEMOE_MXFP4) == 7


@pytest.mark.parametrize("quant,n", [(0, 7), (1, 7), (2, 8), (3, 7), (4, 8), (5, 8)])
def test_every_form_names_its_launches(lib, quant, n):
    # FP8 and the W4A4 forms launch act_quant between w13 and w2
    names = [mm.musemoe_kernel_name(quant, i) for i in range(mm.musemoe_num_kernels(quant))]
    assert len(names) == n
    want = ["router", "pool", "w13"] + (["act_quant"] if n == 8 else []) + \
        ["w2", "finalize", "unpool", "boundary"]
    assert names == want
    assert mm.musemoe_kernel_name(quant, n) == ""


def test_w4a4_workspace_holds_the_rounded_inputs(lib):
    # the W4A4 forms hold both FP4 expert inputs as e2m1 codes and block
    # scales: h [rows, P / 2 + P / 16] in place of the weight format's f16 h
    # operand [rows, P], and w2's input [rows * k, I / 2 + I / 16] on top
    R, P, I, k = 8, 2048, 1024, 8
    d = mm.Dims(max_rows=R, hidden=5120, pooled=P, inter=I, experts=128, top_k=k)
    want = (R * P // 2 + R * P // 16) - R * P * 2 + R * k * (I // 2 + I // 16)
    for w4, a4 in [(mm.MUSEMOE_MXFP4, mm.MUSEMOE_MXFP4_A4), (mm.MUSEMOE_NVFP4, mm.MUSEMOE_NVFP4_A4)]:
        got = mm.musemoe_workspace_bytes(d, a4) - mm.musemoe_workspace_bytes(d, w4)
        assert abs(got - want) <= 4 * 256, (got, want)  # each buffer rounds up to 256 bytes
    assert mm.musemoe_workspace_bytes(d, 6) == 0  # no such form


def test_create_rejects_bad_arguments_before_touching_a_device(lib):
    d = mm.Dims(max_rows=0, hidden=100, pooled=256, inter=128, experts=16, top_k=2)
    c = mm.Config(score=0, route_scale=2.5, norm_eps=1e-6, pre_expert_norm=1)
    with pytest.raises(mm.MuseMoEError) as ei:
        mm.musemoe_create(d, mm.MUSEMOE_MXFP4, c)
    assert ei.value.status == mm.MUSEMOE_EUNSUPPORTED
    assert "max_rows" in str(ei.value) and "hidden 100" in str(ei.value)


def test_create_without_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    d = mm.Dims(max_rows=4, hidden=512, pooled=256, inter=128, experts=16, top_k=2)
    c = mm.Config(score=0, route_scale=2.5, norm_eps=1e-6, pre_expert_norm=1)
    with pytest.raises(mm.MuseMoEError) as ei:
        mm.musemoe_create(d, mm.MUSEMOE_MXFP4, c)
    assert ei.value.status == mm.MUSEMOE_ECUDA
    assert mm.musemoe_last_error(None)


def test_calls_with_null_handle_fail_cleanly(lib):
    assert lib.musemoe_forward(None, None, None, None, None, 1, None) == mm.MUSEMOE_EINVAL
    assert lib.musemoe_poll_health(None) == mm.MUSEMOE_EINVAL
    lib.musemoe_destroy(None)
