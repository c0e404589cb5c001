"""The seeded input generator: determinism, sub-range regeneration and the
value distributions of the block's synthetic workloads. CPU only."""
import numpy as np
import torch

import synth


def test_deterministic_and_subrange_consistent():
    a = synth.random_bytes(7, synth.T_W13, (1000,))
    b = synth.random_bytes(7, synth.T_W13, (1000,))
    assert np.array_equal(a, b)
    assert np.array_equal(synth.random_bytes(7, synth.T_W13, (300,), start=333), a[333:633])
    n = synth.normal_f32(3, synth.T_X, (4097,))
    assert np.array_equal(synth.normal_f32(3, synth.T_X, (101,), start=1001), n[1001:1102])
    assert np.array_equal(synth.normal_f32(3, synth.T_X, (100,), start=2000), n[2000:2100])
    assert not np.array_equal(synth.normal_f32(4, synth.T_X, (64,)), n[:64])
    assert not np.array_equal(synth.normal_f32(3, synth.T_STREAM, (64,)), n[:64])


def test_normal_and_uniform_moments():
    z = synth.normal_f32(11, 99, (400000,)).astype(np.float64)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    zb = torch.from_numpy(synth.normal_bf16(11, 98, (200000,), 1.0, 0.05).view(np.int16)
                          ).view(torch.bfloat16).double().numpy()
    assert abs(zb.mean() - 1) < 0.001 and abs(zb.std() - 0.05) < 0.001
    u = synth.uniform_f32(11, 97, (200000,), -0.1, 0.1)
    assert u.min() >= -0.1 and u.max() < 0.1 and abs(u.mean()) < 0.002


def test_scale_generators():
    s = synth.int_u8(1, 5, (50000,), -8, -4, 127)
    assert set(np.unique(s).tolist()) == {119, 120, 121, 122, 123}
    c = synth.e4m3_pow2(1, 6, (50000,), -6.0, -2.0)
    v = torch.from_numpy(c).view(torch.float8_e4m3fn).double().numpy()
    assert v.min() >= 2.0 ** -6 * 0.999 and v.max() <= 2.0 ** -2 * 1.001


def test_fp8_rows_hit_448():
    codes, scales = synth.fp8_rows(2, 6, 16, 256, 0.05)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert (np.abs(vals).max(axis=1) == 448.0).all()
    w = synth.normal_f32(0, 0, (1,))  # keeps the generator loaded; values unused
    assert w.shape == (1,)
    assert np.all(scales > 0)


def test_workload_shapes_and_hot_experts():
    cfg = synth.CONFIGS["tiny"]
    w = synth.layer_tensors(cfg)
    assert w["w13"].shape == (16, 256, 128) and w["w13_scale"].shape == (16, 256, 8)
    assert w["w2"].shape == (16, 256, 64) and w["w2_scale"].shape == (16, 256, 4)
    assert w["w_pool"].shape == (256, 512) and w["w_unpool"].shape == (512, 256)
    d = synth.dense_tensors(synth.CONFIGS["verify"], 0)
    assert int((d["expert_bias"] == np.float32(0.3)).sum()) == 16
    x, st = synth.activations(cfg)
    assert x.shape == (4, 512) and x.dtype == np.uint16 and st.dtype == np.float32
    e = synth.expert_tensors(cfg, 0, e0=5, ne=2)
    assert np.array_equal(e["w13"], w["w13"][5:7]) and np.array_equal(e["w2_scale"],
                                                                      w["w2_scale"][5:7])
