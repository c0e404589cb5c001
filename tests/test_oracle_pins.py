"""Pins of the oracle against things other than itself: hand-worked closed
forms, library routines for the number formats and norms, invariants of the
routing rule, brute force on tiny experts. CPU only."""
import dataclasses
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle as O
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- formats

def test_bf16_decode_matches_torch():
    bits = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    want = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    got = O.bf16_to_f64(bits)
    finite = np.isfinite(want)
    assert np.array_equal(got[finite], want[finite])
    assert np.array_equal(np.isnan(got), np.isnan(want))


def test_round_bf16_matches_torch_on_fp32_inputs():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.005859375, 3e38, -3.4e38])])
    v = v.astype(np.float32)
    want = torch.from_numpy(v).to(torch.bfloat16).double().numpy()
    got = O.round_bf16(v.astype(np.float64))
    assert np.array_equal(got, want)


def test_round_bf16_ties_to_even_on_exact_midpoints():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties go to the even mantissa (1.0);
    # 1 + 3*2^-8 lies between 1 + 2^-7 (odd) and 1 + 2^-6 (even).
    assert O.round_bf16(1 + 2.0 ** -8) == 1.0
    assert O.round_bf16(1 + 3 * 2.0 ** -8) == 1 + 2.0 ** -6
    assert O.round_bf16(1 + 2.0 ** -8 + 2.0 ** -40) == 1 + 2.0 ** -7
    # a direct fp64 rounding (no detour through fp32, which would double-round)
    assert O.round_bf16(1 + 2.0 ** -8 + 2.0 ** -30) == 1 + 2.0 ** -7


def test_bf16_bits_roundtrip():
    bits = np.arange(0, 0x7F80, 3, dtype=np.uint16)
    assert np.array_equal(O.f64_to_bf16_bits(O.bf16_to_f64(bits)), bits)


def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = O.e4m3_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert O.e4m3_decode(np.array([0x7E]))[0] == 448.0
    assert O.e4m3_decode(np.array([0x01]))[0] == 2.0 ** -9


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(1)
    v = (rng.standard_normal(50000) * 2.0 ** rng.integers(-12, 9, 50000)).astype(np.float32)
    v = v[np.abs(v) <= 448]
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = O.e4m3_encode(v.astype(np.float64))
    # torch keeps the sign of a value that rounds to zero; compare values for zeros
    same = (got == want) | ((O.e4m3_decode(got) == 0) & (O.e4m3_decode(want) == 0))
    assert same.all()


def test_e4m3_encode_saturates():
    assert list(O.e4m3_encode(np.array([448.0, 449.0, 470.0, 1e6, -1e6, -500.0]))) == [
        0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]


def test_e2m1_table_matches_the_minifloat_definition():
    # e2m1: sign bit, 2 exponent bits with bias 1, 1 mantissa bit; exponent
    # field 0 is subnormal with exponent 1 - bias = 0.
    for code in range(16):
        s, e, m = code >> 3, (code >> 1) & 3, code & 1
        mag = 2.0 ** (e - 1) * (1 + m / 2) if e else (m / 2)
        want = -mag if s else mag
        assert O.e2m1_decode(np.array([code]))[0] == want
        assert math.copysign(1, O.e2m1_decode(np.array([code]))[0]) == (-1 if s else 1)


def test_ue8m0_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e8m0fnu).double().numpy()
    got = O.ue8m0_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


def test_fp4_nibble_order():
    # element 2j in the low nibble of byte j
    assert list(O.unpack_fp4(np.array([[0x21, 0xF3]], np.uint8))[0]) == [1, 2, 3, 15]


# ---------------------------------------------------------------- norms

def test_rms_norm_matches_torch():
    rng = np.random.default_rng(2)
    v = rng.standard_normal((5, 64)) * 3
    w = 1 + 0.05 * rng.standard_normal(64)
    want = torch.nn.functional.rms_norm(torch.from_numpy(v), (64,), torch.from_numpy(w),
                                        eps=1e-6).numpy()
    np.testing.assert_allclose(O.rms_norm(v, w, 1e-6), want, rtol=1e-13, atol=0)


def test_rms_norm_invariants():
    rng = np.random.default_rng(3)
    v = rng.standard_normal((3, 100))
    eps = 1e-3
    n = O.rms_norm(v, 1.0, eps)
    ms = (v * v).mean(axis=-1)
    np.testing.assert_allclose((n * n).mean(axis=-1), ms / (ms + eps), rtol=1e-12)
    np.testing.assert_allclose(O.rms_norm(7.5 * v, 1.0, 0.0), O.rms_norm(v, 1.0, 0.0),
                               rtol=1e-12)
    assert np.all(O.rms_norm(np.zeros((1, 8)), 1.0, 1e-6) == 0)


# ---------------------------------------------------------------- routing

def _load_cases():
    with open(os.path.join(GOLDEN, "routing_hand_cases.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _load_cases(), ids=lambda c: c["name"])
def test_routing_hand_cases(case):
    r = O.route(O.round_f32(np.array(case["logits"])), np.array(case["bias"], np.float32),
                case["top_k"], case["route_scale"], case["multiplier"], case["score"],
                case["division_eps"])
    assert r.ids.tolist() == case["ids"]
    np.testing.assert_allclose(r.weights, case["weights"], rtol=2e-7, atol=0)


def _random_logits(seed, b=16, E=32, scale=2.0):
    rng = np.random.default_rng(seed)
    return O.round_f32(rng.standard_normal((b, E)) * scale), rng


@pytest.mark.parametrize("score", ["sigmoid", "softmax"])
@pytest.mark.parametrize("eps", [None, 1e-20, 1e-3])
def test_routing_weights_sum(score, eps):
    logits, rng = _random_logits(4)
    bias = rng.uniform(-0.1, 0.1, 32).astype(np.float32)
    r = O.route(logits, bias, 6, 2.5, 0.5, score, eps)
    rows = np.arange(16)[:, None]
    S = r.scores[rows, r.ids].sum(axis=-1)
    want = 2.5 * S / (S + (np.float32(eps) if eps is not None else 0.0))
    np.testing.assert_allclose(r.weights.sum(axis=-1), want, rtol=1e-6)


def test_routing_ids_unique_and_in_range():
    logits, rng = _random_logits(5, b=64, E=128)
    r = O.route(logits, rng.uniform(-0.1, 0.1, 128).astype(np.float32), 8, 2.5, None,
                "sigmoid", None)
    assert r.ids.dtype == np.int32
    assert ((r.ids >= 0) & (r.ids < 128)).all()
    assert all(len(set(row)) == 8 for row in r.ids.tolist())
    # ids are in descending selection order, and every unselected score is lower
    rows = np.arange(64)[:, None]
    sel = r.selection[rows, r.ids]
    assert (np.diff(sel, axis=-1) <= 0).all()
    mask = np.ones_like(r.selection, dtype=bool)
    mask[rows, r.ids] = False
    assert (r.selection[mask].reshape(64, -1).max(axis=-1) <= sel[:, -1]).all()


def test_bias_changes_selection_never_the_weight_formula():
    logits, rng = _random_logits(6, b=32, E=16)
    b1 = rng.uniform(-0.1, 0.1, 16).astype(np.float32)
    b2 = b1.copy()
    b2[3] += np.float32(0.5)                   # expert 3 becomes much easier to select
    r1 = O.route(logits, b1, 4, 2.5, None, "sigmoid", 1e-20)
    r2 = O.route(logits, b2, 4, 2.5, None, "sigmoid", 1e-20)
    assert (r1.ids != r2.ids).any()            # the bias did move some selections
    same = (r1.ids == r2.ids).all(axis=-1)
    assert same.any()
    np.testing.assert_array_equal(r1.weights[same], r2.weights[same])
    # the weights only ever use the unbiased scores: gather them directly
    rows = np.arange(32)[:, None]
    s = r2.scores[rows, r2.ids]
    np.testing.assert_allclose(r2.weights, 2.5 * s / s.sum(-1, keepdims=True), rtol=1e-6)


def test_uniform_bias_shift_keeps_ids():
    logits, rng = _random_logits(7, b=32, E=32)
    bias = rng.uniform(-0.1, 0.1, 32).astype(np.float32)
    r1 = O.route(logits, bias, 5, 2.5, None, "sigmoid", None)
    r2 = O.route(logits, bias + np.float32(0.25), 5, 2.5, None, "sigmoid", None)
    clear = r1.gap > 1e-5
    np.testing.assert_array_equal(r1.ids[clear], r2.ids[clear])


def test_routing_permutation_equivariance():
    logits, rng = _random_logits(8, b=16, E=32)
    bias = rng.uniform(-0.1, 0.1, 32).astype(np.float32)
    perm = rng.permutation(32)
    r1 = O.route(logits, bias, 4, 2.5, None, "softmax", 1e-6)
    r2 = O.route(logits[:, perm], bias[perm], 4, 2.5, None, "softmax", 1e-6)
    clear = r1.gap > 1e-6
    np.testing.assert_array_equal(perm[r2.ids][clear], r1.ids[clear])
    np.testing.assert_allclose(r2.weights[clear], r1.weights[clear], rtol=1e-6)


def test_scores_match_scipy_and_full_topk_reduces_to_softmax():
    logits, _ = _random_logits(9, b=8, E=16)
    r = O.route(logits, np.zeros(16, np.float32), 16, 2.5, None, "softmax", 1e-6)
    sm = scipy.special.softmax(logits, axis=-1)
    np.testing.assert_allclose(r.scores, sm, rtol=1e-6)
    rows = np.arange(8)[:, None]
    # k = E: the weights are the softmax itself scaled by route_scale / (1 + eps)
    np.testing.assert_allclose(r.weights, 2.5 * sm[rows, r.ids] / (1 + 1e-6), rtol=1e-6)
    rs = O.route(logits, np.zeros(16, np.float32), 3, 1.0, 0.5, "sigmoid", None)
    np.testing.assert_allclose(rs.scores, scipy.special.expit(0.5 * logits), rtol=1e-6)


def test_invalid_score_raises():
    with pytest.raises(ValueError):
        O.route(np.zeros((1, 4)), np.zeros(4, np.float32), 1, 1.0, None, "relu", None)


# ---------------------------------------------------------------- GEMVs

def _bf16(v):
    return O.f64_to_bf16_bits(O.round_bf16(v))


def test_router_logits_one_hot_columns():
    rng = np.random.default_rng(10)
    W = rng.standard_normal((8, 32)).astype(np.float32)
    x = np.zeros((3, 32))
    x[0, 5], x[1, 17], x[2, 31] = 1.0, -2.0, 0.5
    lg = O.router_logits(_bf16(x), W)
    np.testing.assert_array_equal(lg[0], W[:, 5])
    np.testing.assert_array_equal(lg[1], -2.0 * W[:, 17])
    np.testing.assert_array_equal(lg[2], 0.5 * W[:, 31])


def test_pooler_one_hot_without_and_with_norm():
    rng = np.random.default_rng(11)
    Wp = _bf16(rng.standard_normal((16, 24)) * 0.1)
    wn = _bf16(1 + 0.05 * rng.standard_normal(16))
    x = np.zeros((2, 24))
    x[0, 3], x[1, 20] = 1.0, 1.0
    h = O.pre_expert(_bf16(x), Wp, wn, 1e-6, pre_norm=False)
    np.testing.assert_array_equal(h[0], O.bf16_to_f64(Wp[:, 3]))
    np.testing.assert_array_equal(h[1], O.bf16_to_f64(Wp[:, 20]))
    hn = O.pre_expert(_bf16(x), Wp, wn, 1e-6, pre_norm=True)
    col = O.bf16_to_f64(Wp[:, 20])
    want = torch.nn.functional.rms_norm(torch.from_numpy(col), (16,),
                                        torch.from_numpy(O.bf16_to_f64(wn)), eps=1e-6)
    np.testing.assert_array_equal(hn[1], O.round_bf16(want.numpy()))


def test_unpool_one_hot():
    rng = np.random.default_rng(12)
    Wu = _bf16(rng.standard_normal((40, 16)) * 0.1)
    m = np.zeros((1, 16))
    m[0, 9] = 3.0
    np.testing.assert_array_equal(O.unpool(m, Wu)[0], 3.0 * O.bf16_to_f64(Wu[:, 9]))


# ---------------------------------------------------------------- experts

def _decode_nibble_bits(c):
    s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
    mag = 2.0 ** (e - 1) * (1 + m / 2) if e else m / 2
    return -mag if s else mag


def test_mxfp4_dequant_brute_force():
    rng = np.random.default_rng(13)
    t = {"w13": rng.integers(0, 256, (2, 64, 32), dtype=np.uint8),
         "w13_scale": rng.integers(119, 124, (2, 64, 2), dtype=np.uint8),
         "w2": rng.integers(0, 256, (2, 64, 16), dtype=np.uint8),
         "w2_scale": rng.integers(119, 124, (2, 64, 1), dtype=np.uint8)}
    w13, w2 = O.dequant_expert("mxfp4", t, 1)
    for n in range(64):
        for k in range(64):
            byte = int(t["w13"][1, n, k // 2])
            code = byte & 0xF if k % 2 == 0 else byte >> 4
            want = _decode_nibble_bits(code) * 2.0 ** (int(t["w13_scale"][1, n, k // 32]) - 127)
            assert w13[n, k] == want
    assert w2.shape == (64, 32)
    for n in range(64):
        for k in range(32):
            byte = int(t["w2"][1, n, k // 2])
            code = byte & 0xF if k % 2 == 0 else byte >> 4
            assert w2[n, k] == _decode_nibble_bits(code) * 2.0 ** (int(t["w2_scale"][1, n, 0]) - 127)


def test_nvfp4_and_fp8_dequant_brute_force():
    rng = np.random.default_rng(14)
    sf = np.array([0x38, 0x30, 0x01, 0x7E], np.uint8)   # 1, 0.5, 2^-9, 448
    t = {"w13": rng.integers(0, 256, (1, 4, 32), dtype=np.uint8),
         "w13_scale": np.tile(sf, (1, 4, 1)).reshape(1, 4, 4),
         "w13_gscale": np.array([1.25], np.float32),
         "w2": rng.integers(0, 256, (1, 64, 8), dtype=np.uint8),
         "w2_scale": np.full((1, 64, 1), 0x38, np.uint8),
         "w2_gscale": np.array([0.75], np.float32)}
    w13, _ = O.dequant_expert("nvfp4", t, 0)
    sfv = [1.0, 0.5, 2.0 ** -9, 448.0]
    for n in range(4):
        for k in range(64):
            byte = int(t["w13"][0, n, k // 2])
            code = byte & 0xF if k % 2 == 0 else byte >> 4
            assert w13[n, k] == _decode_nibble_bits(code) * sfv[k // 16] * 1.25
    f = {"w13": np.array([[[0x38, 0xB8, 0x7E]]], np.uint8),
         "w13_scale": np.array([[0.5]], np.float32),
         "w2": np.array([[[0x40]]], np.uint8), "w2_scale": np.array([[3.0]], np.float32)}
    w13, w2 = O.dequant_expert("fp8", f, 0)
    assert w13.tolist() == [[0.5, -0.5, 224.0]] and w2.tolist() == [[6.0]]


def _mx_expert(P, I, w13_vals, w2_vals):
    """Pack exact e2m1 values (scale 2^0) into the plain MXFP4 layout."""
    inv = {v: c for c, v in enumerate(O.E2M1[:8])}

    def pack(vals):
        vals = np.asarray(vals, dtype=np.float64)
        codes = np.vectorize(lambda v: inv[abs(v)] | (8 if v < 0 else 0))(vals).astype(np.uint8)
        return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)

    return {"w13": pack(w13_vals)[None], "w13_scale": np.full((1, 2 * I, P // 32), 127, np.uint8),
            "w2": pack(w2_vals)[None], "w2_scale": np.full((1, P, I // 32), 127, np.uint8)}


def test_expert_gate_up_order_and_transposes():
    P, I = 32, 32
    rng = np.random.default_rng(15)
    vals = np.array([0, 0.5, 1, 1.5, 2, -1, -0.5, 3])
    A = rng.choice(vals, (I, P))
    B = rng.choice(vals, (I, P))
    C = rng.choice(vals, (P, I))
    t = _mx_expert(P, I, np.concatenate([A, B]), C)
    h = O.round_bf16(rng.standard_normal((1, P)))
    y = O.expert_outputs(h, np.array([[0]]), "mxfp4", t, I)
    g, u = A @ h[0], B @ h[0]
    a = O.round_bf16(g / (1 + np.exp(-g)) * u)
    np.testing.assert_allclose(y[0, 0], C @ a, rtol=1e-12, atol=1e-12)


def test_silu_matches_torch():
    z = np.linspace(-20, 20, 101)
    np.testing.assert_allclose(O.silu(z), torch.nn.functional.silu(torch.from_numpy(z)).numpy(),
                               rtol=1e-14, atol=1e-300)


def test_fp8_row_quant_maps_amax_to_448():
    rng = np.random.default_rng(16)
    v = O.round_bf16(rng.standard_normal((6, 128)) * 3)
    q, s = O.quantize_rows_e4m3(v)
    back = O.e4m3_decode(q) * s[:, None]
    amax = np.abs(v).max(axis=-1)
    assert (np.abs(O.e4m3_decode(q)).max(axis=-1) == 448.0).all()
    np.testing.assert_allclose(np.abs(back).max(axis=-1), amax, rtol=2 ** -22)
    # e4m3 keeps 4 significant bits: half an ulp is 2^-4 relative (normal range)
    big = np.abs(v) > amax[:, None] * 2.0 ** -6
    assert (np.abs(back - v)[big] <= np.abs(v)[big] * 2.0 ** -4 * (1 + 1e-6)).all()
    q0, s0 = O.quantize_rows_e4m3(np.zeros((1, 8)))
    assert s0[0] == 0 and (q0 == 0).all()


# ---------------------------------------------------------------- tail and boundary

def test_single_route_closed_form():
    rng = np.random.default_rng(17)
    y = rng.standard_normal((3, 1, 64))
    wpost = _bf16(1 + 0.05 * rng.standard_normal(64))
    w = np.array([[2.5 * 0.7 / (0.7 + 1e-20)]] * 3)
    out = O.finalize(y, w, wpost, 1e-6)
    want = O.round_bf16(w[:, 0:1] * O.rms_norm(y[:, 0], O.bf16_to_f64(wpost), 1e-6))
    np.testing.assert_array_equal(out, want)


def test_identical_experts_make_the_output_independent_of_routing():
    cfg_rng = np.random.default_rng(18)
    P, I, E, H = 64, 32, 6, 96
    codes13 = cfg_rng.integers(0, 256, (1, 2 * I, P // 2), dtype=np.uint8)
    codes2 = cfg_rng.integers(0, 256, (1, P, I // 2), dtype=np.uint8)
    t = {"w13": np.repeat(codes13, E, 0), "w13_scale": np.full((E, 2 * I, P // 32), 121, np.uint8),
         "w2": np.repeat(codes2, E, 0), "w2_scale": np.full((E, P, I // 32), 122, np.uint8)}
    h = O.round_bf16(cfg_rng.standard_normal((4, P)))
    ids_a = np.array([[0, 1], [2, 3], [4, 5], [1, 0]])
    ids_b = np.array([[5, 4], [0, 2], [3, 1], [2, 5]])
    ya = O.expert_outputs(h, ids_a, "mxfp4", t, I)
    yb = O.expert_outputs(h, ids_b, "mxfp4", t, I)
    np.testing.assert_array_equal(ya, yb)
    wpost = _bf16(np.ones(P))
    S = np.array([[0.6, 0.3]] * 4)
    wts = O.round_f32(2.5 * S / (S.sum(-1, keepdims=True) + 1e-20))
    out = O.finalize(ya, wts, wpost, 1e-6)
    n = O.rms_norm(ya[:, 0], 1.0, 1e-6)
    np.testing.assert_allclose(out, O.round_bf16(wts.sum(-1, keepdims=True) * n), rtol=2 ** -7)
    assert H  # dims documented above


def test_boundary_linearity_and_zero_gate():
    rng = np.random.default_rng(19)
    u = rng.standard_normal((2, 48))
    stream = rng.standard_normal((2, 48)).astype(np.float32)
    wf = _bf16(1 + 0.05 * rng.standard_normal(48))
    wn = _bf16(1 + 0.05 * rng.standard_normal(48))
    s1, out = O.boundary(u, stream, wf, 0.75, wn, 1e-6)
    add = O.rms_norm(u, O.bf16_to_f64(wf), 1e-6)
    np.testing.assert_allclose(s1 - stream, 0.75 * add, atol=4 * 2.0 ** -24 * np.abs(s1).max())
    s0, _ = O.boundary(u, stream, wf, 0.0, wn, 1e-6)
    np.testing.assert_array_equal(s0, stream.astype(np.float64))
    want = torch.nn.functional.rms_norm(torch.from_numpy(s1), (48,),
                                        torch.from_numpy(O.bf16_to_f64(wn)), eps=1e-6).numpy()
    np.testing.assert_array_equal(out, O.round_bf16(want))


def test_attention_boundary_hand_worked():
    # partial [1, -1, 1, -1] has RMS 1 (eps 0): the weightless norm leaves it;
    # stream 0.5 + 2 * partial = [2.5, -1.5, 2.5, -1.5], RMS sqrt(4.25);
    # 2.5 / sqrt(4.25) = 1.21268 -> bf16 1.2109375 (27/128 above 1, the next
    # step is 28/128 = 1.21875); -1.5 / sqrt(4.25) = -0.72761 -> bf16
    # -0.7265625 (186/256; 187/256 = 0.73047 is farther)
    partial = np.array([[0x3F80, 0xBF80, 0x3F80, 0xBF80]], dtype=np.uint16)
    stream = np.full((1, 4), 0.5, dtype=np.float32)
    w = np.full(4, 0x3F80, dtype=np.uint16)
    s_new, out = O.attention_boundary(partial, stream, 2.0, w, 0.0)
    np.testing.assert_array_equal(s_new, [[2.5, -1.5, 2.5, -1.5]])
    np.testing.assert_array_equal(out, [[1.2109375, -0.7265625, 1.2109375, -0.7265625]])


def test_attention_boundary_norm_is_weightless_and_scale_free():
    rng = np.random.default_rng(23)
    partial = _bf16(rng.standard_normal((3, 64)))
    w = _bf16(1 + 0.05 * rng.standard_normal(64))
    zero = np.zeros((3, 64), dtype=np.float32)
    # gate 1 onto a zero stream: the stream becomes the normalized partial,
    # mean square 1 per row (eps 0), whatever the pre_ffn_norm weight
    s_new, _ = O.attention_boundary(partial, zero, 1.0, w, 0.0)
    np.testing.assert_allclose(np.mean(s_new * s_new, axis=1), 1.0, rtol=1e-6)
    # x4 is exact in bf16 and the norm removes it
    p4 = O.f64_to_bf16_bits(4.0 * O.bf16_to_f64(partial))
    stream = rng.standard_normal((3, 64)).astype(np.float32)
    a = O.attention_boundary(partial, stream, 0.6, w, 0.0)
    b = O.attention_boundary(p4, stream, 0.6, w, 0.0)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_attention_boundary_zero_gate_and_unit_weight_ffn_form():
    rng = np.random.default_rng(29)
    partial = _bf16(rng.standard_normal((2, 48)))
    stream = rng.standard_normal((2, 48)).astype(np.float32)
    w = _bf16(1 + 0.05 * rng.standard_normal(48))
    s0, out0 = O.attention_boundary(partial, stream, 0.0, w, 1e-6)
    np.testing.assert_array_equal(s0, stream.astype(np.float64))
    want = torch.nn.functional.rms_norm(torch.from_numpy(stream.astype(np.float64)), (48,),
                                        torch.from_numpy(O.bf16_to_f64(w)), eps=1e-6).numpy()
    np.testing.assert_array_equal(out0, O.round_bf16(want))
    # the FFN boundary with a unit post-norm weight and the bf16 input as u
    ones = np.full(48, 0x3F80, dtype=np.uint16)
    sa, oa = O.attention_boundary(partial, stream, 0.8, w, 1e-6)
    sf, of = O.boundary(O.bf16_to_f64(partial), stream, ones, 0.8, w, 1e-6)
    np.testing.assert_array_equal(sa, sf)
    np.testing.assert_array_equal(oa, of)


def test_bf16_experts_equal_their_exact_mxfp4_twins():
    # MXFP4 values are exact in bf16: BF16 experts holding the dequantized
    # MXFP4 weights give the same expert outputs through their own dequant
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], experts=4, seed=41)
    t = synth.expert_tensors(cfg, 0)
    tb = {}
    for k in ("w13", "w2"):
        vals = np.stack([O.dequant_expert("mxfp4", t, e)[0 if k == "w13" else 1] for e in range(4)])
        tb[k] = O.f64_to_bf16_bits(vals)
        np.testing.assert_array_equal(O.bf16_to_f64(tb[k]), vals)
    rng = np.random.default_rng(43)
    h = O.round_bf16(rng.standard_normal((3, cfg.pooled)))
    ids = np.array([[0, 3], [2, 1], [3, 3]])
    y4 = O.expert_outputs(h, ids, "mxfp4", t, cfg.inter)
    yb = O.expert_outputs(h, ids, "bf16", tb, cfg.inter)
    np.testing.assert_array_equal(y4, yb)
    with pytest.raises(ValueError):
        O.dequant_expert("int4", t, 0)


# ---------------------------------------------------------------- online MXFP4 rounding

def _blocks(rows):
    return O.f64_to_bf16_bits(np.asarray(rows, dtype=np.float64))


def test_quantize_mxfp4_hand_worked():
    # amax 6: floor(log2 6) = 2, scale 2^0 (UE8M0 127); 6 -> code 7, -6 -> 0xF
    b = np.zeros((1, 32)); b[0, 0], b[0, 1] = 6.0, -6.0
    packed, scale = O.quantize_mxfp4(_blocks(b))
    assert scale.tolist() == [[127]] and packed[0, 0] == 0xF7 and not packed[0, 1:].any()
    # amax 7 keeps scale 2^0; ties go to the even code, 7 saturates at 6:
    # 0.25->0, 0.75->1.0 (code 2), 1.25->1.0, 1.75->2.0 (4), 2.5->2.0,
    # 3.5->4.0 (6), 5.0->4.0, 7.0->6.0 (7); 0.3->0.5 (1), -2.9->-3.0 (0xD)
    row = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 0.3, -2.9] + [0.0] * 22
    packed, scale = O.quantize_mxfp4(_blocks([row]))
    codes = O.unpack_fp4(packed)[0, :10].tolist()
    assert scale.tolist() == [[127]]
    assert codes == [0, 2, 2, 4, 4, 6, 6, 7, 1, 0xD]
    # all ones: amax 1 -> scale 2^-2 (UE8M0 125), 1 / 2^-2 = 4 -> code 6
    packed, scale = O.quantize_mxfp4(_blocks(np.ones((1, 32))))
    assert scale.tolist() == [[125]] and (O.unpack_fp4(packed) == 6).all()
    # a zero block takes 2^0; -0.0 keeps its sign bit
    z = np.zeros((1, 32)); z[0, 3] = -0.0
    packed, scale = O.quantize_mxfp4(_blocks(z))
    assert scale.tolist() == [[127]] and O.unpack_fp4(packed)[0, 3] == 8
    # a subnormal amax (2^-130): exponent -132 clamps to -126 (UE8M0 1), the
    # element is 2^-4 of the scale and rounds to 0
    t = np.zeros((1, 32)); t[0, 5] = 2.0 ** -130
    packed, scale = O.quantize_mxfp4(_blocks(t))
    assert scale.tolist() == [[1]] and not packed.any()


def test_quantize_mxfp4_is_nearest_and_scale_in_range():
    rng = np.random.default_rng(31)
    w = _bf16(0.02 * rng.standard_normal((6, 256)))
    packed, scale = O.quantize_mxfp4(w)
    v = O.bf16_to_f64(w).reshape(6, 8, 32)
    sc = O.ue8m0_decode(scale)[..., None]
    a = np.abs(v) / sc
    assert (a.max(axis=-1) >= 4).all() and (a.max(axis=-1) < 8).all()
    q = np.abs(O.e2m1_decode(O.unpack_fp4(packed))).reshape(6, 8, 32)
    grid = O.E2M1[:8]
    nearest = np.abs(a[..., None] - grid).min(axis=-1)
    np.testing.assert_array_equal(np.abs(a - q), nearest)  # no nearer grid value exists
    assert (np.sign(O.e2m1_decode(O.unpack_fp4(packed))).reshape(6, 8, 32) * np.sign(v) >= 0).all()


def test_quantize_mxfp4_round_trips_representable_blocks():
    rng = np.random.default_rng(37)
    codes = rng.integers(0, 16, size=(4, 128)).astype(np.uint8)
    codes[:, ::32] = 7  # one element of magnitude 6 per block fixes the scale
    exps = rng.integers(110, 140, size=(4, 4)).astype(np.uint8)
    vals = O.e2m1_decode(codes) * np.repeat(O.ue8m0_decode(exps), 32, axis=1)
    packed, scale = O.quantize_mxfp4(O.f64_to_bf16_bits(vals))
    np.testing.assert_array_equal(scale, exps)
    # codes round-trip bit for bit (-0.0 included: its sign bit is kept)
    np.testing.assert_array_equal(O.unpack_fp4(packed), codes)


# ---------------------------------------------------------------- near-tie rounding rule

def test_round_bf16_near_takes_only_values_inside_the_band():
    row = np.array([[1.0 + 2.0 ** -8, 1.0 + 2.0 ** -6 + 1e-3, 3e-7, 1.0]])
    # the first element is exactly a rounding midpoint: either neighbour is valid
    near = np.array([[1.0 + 2.0 ** -7, 1.0 + 2.0 ** -6, 2.9e-7, 1.0]])
    out, n = O.round_bf16_near(row, near, band=2.0 ** -16)
    assert out[0, 0] == 1.0 + 2.0 ** -7 and n >= 1
    # the second is far from a midpoint: the other neighbour is refused
    assert out[0, 1] == O.round_bf16(row[0, 1])
    # a near-zero element: any bf16 value within band * RMS(row) is accepted
    assert out[0, 2] == 2.9e-7
    far = np.array([[1.0 + 2.0 ** -8, 1.0 + 2.0 ** -6 + 1e-3, 5e-4, 1.0]])
    out2, _ = O.round_bf16_near(row, far, band=2.0 ** -16)
    assert out2[0, 2] == O.round_bf16(3e-7)
    # without a hint it is plain round-to-nearest-even
    out3, n3 = O.round_bf16_near(row)
    assert n3 == 0 and np.array_equal(out3, O.round_bf16(row))


# ---------------------------------------------------------------- W4A4 activations

def _nv_expect(codes):
    c = np.asarray(codes, dtype=np.uint8)
    return (c[0::2] | (c[1::2] << 4)).astype(np.uint8)


def test_quantize_act_nvfp4_hand_worked():
    # amax 6 -> scale e4m3(1.0) = 0x38; every e2m1 midpoint goes to the even code
    a = [6, -3, 1.5, 0.5, 0, 2, -4, 1, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -6]
    ca = [7, 13, 3, 1, 0, 4, 14, 2, 0, 2, 2, 4, 4, 6, 6, 15]
    # amax 7 -> 7/6 = 1.1667 -> e4m3 1.125 (0x39); 7/1.125 = 6.22 saturates at 6;
    # 1.125 -> 1 (code 2); -0.5625 -> 0.5 (code 9)
    b = [7, 1.125, -0.5625] + [0] * 13
    cb = [7, 2, 9] + [0] * 13
    # all zero with one -0: scale 0, the sign bit kept
    c = [0, -0.0] + [0] * 14
    cc = [0, 8] + [0] * 14
    # amax 2944 -> 490.7 saturates at 448 (0x7E); 2944/448 = 6.6 -> 6; 448 -> 1
    d = [2944, 448] + [0] * 14
    cd = [7, 2] + [0] * 14
    # amax 2^-12 -> 2^-12/6 below half the smallest e4m3 subnormal: scale 0
    e = [2.0 ** -12, -(2.0 ** -13)] + [0] * 14
    ce = [0, 8] + [0] * 14
    # amax 3 * 2^-8 -> exactly 2^-9, the smallest subnormal (0x01); 2^-10 -> 0.5
    f = [3 * 2.0 ** -8, 2.0 ** -10] + [0] * 14
    cf = [7, 1] + [0] * 14
    # the largest finite bf16: scale 448, a quotient near 7.6e35 saturates to 6
    g = [3.3895313892515355e38, -1.0] + [0] * 14
    cg = [7, 8] + [0] * 14
    rows = np.array([a + b + c + d + e + f + g], dtype=np.float64)
    packed, sc = O.quantize_act_nvfp4(rows)
    want = np.concatenate([_nv_expect(x) for x in (ca, cb, cc, cd, ce, cf, cg)])
    np.testing.assert_array_equal(packed[0], want)
    np.testing.assert_array_equal(sc[0], np.array([0x38, 0x39, 0x00, 0x7E, 0x00, 0x01, 0x7E],
                                                  np.uint8))
    vals = O.fp4_activation(rows, "nvfp4")[0]
    np.testing.assert_array_equal(vals[16:19], [6.75, 1.125, -0.5625])
    assert vals[48] == 6 * 448.0 and vals[80] == 6 * 2.0 ** -9


def _e4m3_table():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().double().numpy()


def test_quantize_act_nvfp4_brute_force():
    # every scale is the nearest finite non-negative e4m3 value to fp32(amax/6)
    # (ties to the even code, saturating), every code the nearest e2m1
    # magnitude to fp32(|v| / scale) (ties to the even code), searched over all
    tab = _e4m3_table()
    pos = np.arange(127)  # finite codes 0x00..0x7E
    rng = np.random.default_rng(53)
    mags = 2.0 ** rng.integers(-14, 12, size=(48, 1))
    v = O.round_bf16(rng.standard_normal((48, 16)) * mags)
    packed, sc = O.quantize_act_nvfp4(v)
    codes = O.unpack_fp4(packed)
    for r in range(v.shape[0]):
        t = np.float32(np.abs(v[r]).max()) / np.float32(6.0)
        dist = np.abs(tab[pos] - float(t))
        best = pos[dist == dist.min()]
        s = best[0] if len(best) == 1 else best[best % 2 == 0][0]
        if float(t) > 448.0:
            s = 0x7E
        assert sc[r, 0] == s, (r, sc[r, 0], s)
        sf = tab[s]
        for j in range(16):
            q = 0.0 if sf == 0 else float(np.float32(abs(v[r, j])) / np.float32(sf))
            d = np.abs(O.E2M1[:8] - q)
            m = np.nonzero(d == d.min())[0]
            mc = m[0] if len(m) == 1 else m[m % 2 == 0][0]
            assert codes[r, j] == (mc | (8 if np.signbit(v[r, j]) else 0)), (r, j)


def test_fp4_activation_round_trips_representable_blocks():
    rng = np.random.default_rng(59)
    mv = rng.choice(O.E2M1[1:8], size=(6, 32)) * rng.choice([-1.0, 1.0], size=(6, 32))
    # MXFP4: a block whose amax is 6 * 2^e holds e2m1 multiples of 2^e exactly
    ex = rng.integers(-6, 6, size=(6, 1))
    mx = mv.copy()
    mx[:, 0] = 6.0
    mx = mx * 2.0 ** ex
    np.testing.assert_array_equal(O.fp4_activation(mx, "mxfp4"), mx)
    # NVFP4: amax = 6 * s with s an e4m3 value gives the scale s back
    s = np.array([1.0, 0.5, 1.125, 2.0 ** -9, 448.0, 13.0])[:, None]
    nv = mv[:, :16].copy()
    nv[:, 3] = -6.0
    nv = nv * s
    np.testing.assert_array_equal(O.fp4_activation(nv, "nvfp4"), nv)


@pytest.mark.parametrize("fmt", ["mxfp4", "nvfp4"])
def test_w4a4_expert_outputs_one_hot(fmt):
    # one-hot experts: gate_i = h[i], up_i = h[I + i] and y[p] = a[p] (p < I), so
    # y is the FP4 rounding of bf16(silu(hq[i]) * hq[I + i]) with hq the FP4
    # rounding of h: both expert inputs rounded, at the format's block size
    P, I = 64, 32
    w13 = np.zeros((1, 2 * I, P), np.uint8)
    for i in range(2 * I):
        w13[0, i, i] = 2  # e2m1 1.0
    w2 = np.zeros((1, P, I), np.uint8)
    for p in range(I):
        w2[0, p, p] = 2
    pk = lambda c: (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)
    t = {"w13": pk(w13), "w2": pk(w2)}
    if fmt == "mxfp4":
        t["w13_scale"] = np.full((1, 2 * I, P // 32), 127, np.uint8)
        t["w2_scale"] = np.full((1, P, I // 32), 127, np.uint8)
    else:
        t["w13_scale"] = np.full((1, 2 * I, P // 16), 0x38, np.uint8)
        t["w2_scale"] = np.full((1, P, I // 16), 0x38, np.uint8)
        t["w13_gscale"] = np.ones(1, np.float32)
        t["w2_gscale"] = np.ones(1, np.float32)
    rng = np.random.default_rng(61)
    h = O.round_bf16(rng.standard_normal((2, P)) * np.array([[1.0], [0.03]]))
    ids = np.zeros((2, 1), np.int64)
    y = O.expert_outputs(h, ids, fmt + "_a4", t, I)[:, 0]

    def fp4(v, block):  # brute force over the block's scale and the 8 magnitudes
        out = np.empty_like(v)
        tab = _e4m3_table()
        for r in range(v.shape[0]):
            for b0 in range(0, v.shape[1], block):
                x = v[r, b0:b0 + block]
                amax = np.abs(x).max()
                if block == 32:
                    sf = 2.0 ** (np.floor(np.log2(amax)) - 2) if amax > 0 else 1.0
                    q = np.abs(x) / sf
                else:
                    t6 = float(np.float32(amax) / np.float32(6.0))
                    fin = tab[:127]
                    dd = np.abs(fin - t6)
                    cands = np.nonzero(dd == dd.min())[0]
                    sf = fin[cands[0] if len(cands) == 1 else cands[cands % 2 == 0][0]]
                    q = (np.abs(x).astype(np.float32) / np.float32(sf)).astype(np.float64) \
                        if sf > 0 else np.zeros_like(x)
                d = np.abs(O.E2M1[:8][None, :] - q[:, None])
                pick = []
                for row in d:
                    m = np.nonzero(row == row.min())[0]
                    pick.append(m[0] if len(m) == 1 else m[m % 2 == 0][0])
                out[r, b0:b0 + block] = np.sign(x) * O.E2M1[np.array(pick)] * sf
        return out

    blk = 32 if fmt == "mxfp4" else 16
    hq = fp4(h, blk)
    g, u = hq[:, :I], hq[:, I:]
    a = torch.tensor(g / (1 + np.exp(-g)) * u).to(torch.bfloat16).double().numpy()
    want = np.zeros((2, P))
    want[:, :I] = fp4(a, blk)
    np.testing.assert_array_equal(y, want)
    # and neither input is left unrounded
    assert not np.array_equal(hq, h) and not np.array_equal(want[:, :I], a)


def _e4m3_nearest_brute(v):
    """e4m3 value nearest each element of v (fp64), searched over every finite
    code; ties to the even code; beyond the largest finite value, 448."""
    tab = _e4m3_table()
    fin = tab[:127]  # 0x00..0x7E: the non-negative finite values
    out = np.empty_like(v)
    for i, x in np.ndenumerate(v):
        a = abs(x)
        if a >= 448.0:
            m = 448.0
        else:
            d = np.abs(fin - a)
            c = np.nonzero(d == d.min())[0]
            m = fin[c[0] if len(c) == 1 else c[c % 2 == 0][0]]
        out[i] = math.copysign(m, x)
    return out


def test_fp8_expert_outputs_permuted_one_hot():
    # permuted one-hot FP8 experts with a distinct fp32 scale per output row:
    # gu[i] = s13[i] * hq[pi(i)], y[p] = s2[p] * aq[p] (p < I), where hq / aq
    # are h per token and a per route requantized to e4m3 with their own
    # dynamic scale fp32(amax / 448) (the W8A8 reading of both expert inputs).
    # A scale applied per column (transposed), or an activation that skips its
    # requantization, fails against this brute force.
    P, I = 64, 16
    rng = np.random.default_rng(67)
    pi = rng.permutation(P)[:2 * I]
    w13 = np.zeros((1, 2 * I, P), np.uint8)
    w13[0, np.arange(2 * I), pi] = 0x38  # e4m3 1.0
    w2 = np.zeros((1, P, I), np.uint8)
    w2[0, np.arange(I), np.arange(I)] = 0x38
    s13 = (0.5 + np.arange(2 * I) / 37.0).astype(np.float32)
    s2 = (0.75 + np.arange(P) / 53.0).astype(np.float32)
    t = {"w13": w13, "w13_scale": s13[None], "w2": w2, "w2_scale": s2[None]}
    h = O.round_bf16(rng.standard_normal((3, P)) * np.array([[1.0], [0.02], [40.0]]))
    ids = np.zeros((3, 1), np.int64)
    y = O.expert_outputs(h, ids, "fp8", t, I)[:, 0]

    def requant(v):
        out = np.empty_like(v)
        for r in range(v.shape[0]):
            s = float(np.float32(np.abs(v[r]).max() / 448.0))
            q = (v[r].astype(np.float32) / np.float32(s)).astype(np.float64)
            out[r] = _e4m3_nearest_brute(q) * s
        return out

    hq = requant(h)
    gu = hq[:, pi] * s13.astype(np.float64)
    g, u = gu[:, :I], gu[:, I:]
    a = torch.tensor(g / (1 + np.exp(-g)) * u).to(torch.bfloat16).double().numpy()
    aq = requant(a)
    want = np.zeros((3, P))
    want[:, :I] = aq * s2[:I].astype(np.float64)
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=0)
    # the planted mistakes differ from it
    skip_a = np.zeros((3, P))
    skip_a[:, :I] = a * s2[:I].astype(np.float64)
    assert np.abs(skip_a - want).max() > 1e-3 * np.abs(want).max()
    assert not np.allclose(hq[:, pi] * s13[::-1].astype(np.float64), gu)  # scales on other rows
    assert not np.array_equal(hq, h) and not np.array_equal(aq, a)
