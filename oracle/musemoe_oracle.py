"""CPU oracle of the MuseSpark1x MoE decode block (numpy, float64).

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this module. The
library's CUDA path never calls it, and it shares no code with that path.

It is a plain, slow, step-by-step restatement of what the pages fix:

* router GEMV and routing rule -- page "vllm.models.muse_spark.amd.muse_moe_runner",
  class MuseSpark1xRouter (its docstring and ``_compute_routing_native``,
  which the page presents as the torch reference of the routing kernel);
* pooler + pre_expert_norm, routed experts, tail, unpooler -- page
  "vllm.models.muse_spark.nvidia.specialized_decode.runtime.providers",
  MoEProvider docstring and RoutedMoE.run;
* post-expert norm before the router weighting, weighted sum -- page
  "vllm.models.muse_spark.amd.muse_moe_runner", MuseSparkTopKWeightAndReduce.apply
  (the unfused branch: norm to fp32, multiply by topk_weights, sum over k);
* routed experts with unit weights (router weighting only after the norm) --
  same page, MuseSparkAiterExperts.apply / ``_unit_weights``;
* MXFP4 expert tensor shapes -- page "vllm.models.muse_spark.amd.mono.decoder",
  MonoDims.expert_shapes;
* FFN boundary (post_ffn_norm, gated add into the fp32 stream in place, next
  pre-norm to bf16) -- providers page, BoundaryProvider docstring;
* attention boundary before the block (weightless post_attn_norm, gated add,
  pre_ffn_norm to bf16) -- providers page, AttentionBoundaryProvider
  docstring, and decoder page (post_attn_norm has no weight).
* online rounding of BF16 expert weights to MXFP4 -- page
  "vllm.models.muse_spark.amd.muse_moe_runner", _quantize_experts_to_mxfp4.
* W4A4 expert inputs: dynamic MXFP4 activations (muse_moe_runner page, the
  Quark w_mxfp4_a_mxfp4 scheme) and the NVFP4 expert input (providers page,
  ExpertsInput: e2m1 codes with e4m3 block scales per 16).

Every value is float64 unless a rounding is named. The rounding points are
the storage dtypes the pages show: fp32 router logits and routing scores
(the routing recipe runs on fp32 tensors), bf16 ``h`` and bf16 MoE
activations (decoder page, _K5Bucket buffers ``h`` bf16; mono page,
maybe_attach_mono, which keeps the MoE activations in bf16), bf16 ``moe_out`` (providers
page, RoutedMoE buffers), fp32 ``stream`` and bf16 ``out`` (BoundaryProvider).
Where the pages are silent the module states the reading it takes.

Inputs use the storage formats: bf16 tensors are uint16 bit patterns, fp32
tensors are float32, quantized expert tensors are uint8 codes (plus fp32
scales where the format has them).
"""
from __future__ import annotations

import dataclasses

import numpy as np

# --------------------------------------------------------------------------
# Number formats
# --------------------------------------------------------------------------


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float64 (bf16 is the top half of an fp32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def round_f32(v) -> np.ndarray:
    """Round float64 values to float32 (IEEE round to nearest even)."""
    return np.asarray(v, dtype=np.float64).astype(np.float32).astype(np.float64)


def _round_minifloat(v, mant_bits: int, min_exp: int) -> np.ndarray:
    """Round to the nearest value with `mant_bits` fraction bits in the binade
    of v (never below the binade 2^min_exp, which gives the subnormal step),
    ties to even. Overflow is left to the caller."""
    v = np.asarray(v, dtype=np.float64)
    _, e = np.frexp(v)                       # v = f * 2^e, |f| in [0.5, 1)
    binade = np.maximum(e - 1, min_exp)      # floor(log2|v|), clamped
    step = np.ldexp(1.0, binade - mant_bits)
    return np.rint(v / step) * step          # np.rint rounds half to even


def round_bf16(v) -> np.ndarray:
    """Round float64 values to bfloat16 (8 significant bits, fp32 exponent
    range, round to nearest even); overflow gives +-inf."""
    r = _round_minifloat(v, 7, -126)
    big = np.abs(r) > 3.3895313892515355e38
    return np.where(big, np.copysign(np.inf, r), r)


# Width of the band, relative to the RMS of the row, inside which a rounding
# decision counts as a near tie (a bound on the fp32 accumulation error of
# the dot products and norms that feed the rounding points).
NEAR_TIE_BAND = 2.0 ** -16


def round_bf16_near(v, near=None, band=NEAR_TIE_BAND):
    """round_bf16 with the near-tie rule of the rounding decision.

    ``near`` holds another computation's bf16 values of the same quantity.
    Where such a value is the bf16 rounding of some value within
    ``band * RMS(row of v)`` of v, the rounding decision is a near tie (both
    results are correct to working precision) and ``near`` is taken;
    everywhere else the result is round_bf16(v). Returns (values, number of
    elements taken from ``near`` that differ from round_bf16(v)).
    """
    r = round_bf16(v)
    if near is None:
        return r, 0
    v = np.asarray(v, dtype=np.float64)
    near = np.asarray(near, dtype=np.float64)
    d = band * np.sqrt(np.mean(v * v, axis=-1, keepdims=True))
    ok = (near >= round_bf16(v - d)) & (near <= round_bf16(v + d))
    return np.where(ok, near, r), int(np.count_nonzero(ok & (near != r)))


def f64_to_bf16_bits(v) -> np.ndarray:
    """bf16-representable float64 values -> their bit patterns."""
    f = np.asarray(v, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


# OCP MX e2m1: sign bit 3, two exponent bits (bias 1), one mantissa bit.
E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                 -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


def unpack_fp4(packed: np.ndarray) -> np.ndarray:
    """[..., K/2] bytes -> [..., K] 4-bit codes; element 2j sits in the low
    nibble of byte j (reading: the pages pack two e2m1 codes into each byte
    but fix no order)."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), np.uint8)
    out[..., 0::2] = p & 0x0F
    out[..., 1::2] = p >> 4
    return out


def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    return E2M1[np.asarray(codes, dtype=np.uint8) & 0x0F]


def quantize_mxfp4(w_bf16: np.ndarray):
    """Round bf16 weights [..., cols] to packed OCP MXFP4: the online rounding
    of BF16 experts on load (page "vllm.models.muse_spark.amd.muse_moe_runner",
    _quantize_experts_to_mxfp4, applied to every decoder layer but the first
    and the last per _online_mxfp4_applies).

    Reading (the page names OCP MXFP4 and a library routine but prints no
    formula): per block of 32 consecutive elements along cols, the shared
    scale is 2^(floor(log2(amax)) - 2), 2 being the largest e2m1 exponent, so
    that amax / scale lies in [4, 8); its exponent is clamped to [-126, 127]
    (UE8M0 codes 1..254, those the kernel layout accepts); an all-zero block
    takes 2^0. Each element becomes the e2m1 magnitude nearest |v| / scale,
    ties to the even code (mantissa bit 0), which saturates at 6; the sign
    bit is kept (a negative value that rounds to 0 gives code 0x8).

    Returns (codes uint8 [..., cols/2], element 2j in the low nibble of byte
    j; scales uint8 [..., cols/32])."""
    v = bf16_to_f64(w_bf16)
    cols = v.shape[-1]
    assert cols % 32 == 0
    blk = v.reshape(v.shape[:-1] + (cols // 32, 32))
    amax = np.abs(blk).max(axis=-1)
    _, ex = np.frexp(amax)  # amax = m * 2^ex, m in [0.5, 1): floor(log2) = ex - 1
    e = np.where(amax > 0, ex - 1 - 2, 0)
    e = np.clip(e, -126, 127)
    a = np.abs(blk) / np.ldexp(1.0, e)[..., None]  # exact: a power of two
    mags = E2M1[:8]
    d = np.abs(a[..., None] - mags)
    best = d.min(axis=-1, keepdims=True)
    cand = d == best
    # among equally near magnitudes (a tie: at most two) take the even code
    even = cand & ((np.arange(8) & 1) == 0)
    code = np.where(even.any(axis=-1), np.argmax(even, axis=-1), np.argmax(cand, axis=-1))
    code = code.astype(np.uint8) | (np.signbit(blk).astype(np.uint8) << 3)
    codes = code.reshape(v.shape)
    packed = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
    return packed, (e + 127).astype(np.uint8)


def ue8m0_decode(s: np.ndarray) -> np.ndarray:
    """UE8M0 scale byte -> 2^(s - 127); 0xFF is NaN."""
    s = np.asarray(s, dtype=np.int64)
    return np.where(s == 255, np.nan, np.ldexp(1.0, s - 127))


def _e4m3_value(c: np.ndarray) -> np.ndarray:
    """OCP float8 e4m3fn: sign, 4 exponent bits (bias 7), 3 mantissa bits, no
    infinities, S.1111.111 is NaN, exponent field 0 is subnormal."""
    c = np.asarray(c, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    ex = (c >> 3) & 0xF
    m = c & 0x7
    normal = np.ldexp(1.0 + m / 8.0, ex - 7)
    sub = np.ldexp(m / 8.0, -6)
    val = sign * np.where(ex == 0, sub, normal)
    return np.where((c & 0x7F) == 0x7F, np.nan, val)


_E4M3_TABLE = _e4m3_value(np.arange(256))


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """e4m3fn codes -> float64 (a lookup in the table of all 256 codes)."""
    return _E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(v) -> np.ndarray:
    """float64 values -> e4m3fn codes, round to nearest even, saturating to
    +-448 (the "satfinite" conversion)."""
    v = np.asarray(v, dtype=np.float64)
    r = _round_minifloat(np.abs(v), 3, -6)
    r = np.minimum(r, 448.0)
    _, e = np.frexp(r)
    binade = e - 1
    normal = r >= 2.0 ** -6
    ex_field = np.where(normal, binade + 7, 0)
    mant = np.where(normal, np.rint(np.ldexp(r, 3 - binade)) - 8, np.rint(r * 512.0))
    code = (ex_field << 3) | mant.astype(np.int64)
    sign = np.signbit(v).astype(np.int64) << 7
    return (code | sign).astype(np.uint8)


# --------------------------------------------------------------------------
# Norms
# --------------------------------------------------------------------------


def rms_norm(v: np.ndarray, w, eps: float) -> np.ndarray:
    """RMSNorm over the last axis, weight applied after normalization:
    v / sqrt(mean(v^2) + eps) * w. (Reading: the pages name the MuseSpark1x
    RMSNorm variants but not their formula; this is the plain form with the
    effective bf16 weight of decoder page, effective_norm_weight.)"""
    v = np.asarray(v, dtype=np.float64)
    ms = np.mean(v * v, axis=-1, keepdims=True)
    return v / np.sqrt(ms + eps) * w


# --------------------------------------------------------------------------
# Router and routing rule
# --------------------------------------------------------------------------


def router_logits(x_bf16: np.ndarray, w_router: np.ndarray) -> np.ndarray:
    """fp32 GateLinear: [b, H] bf16 x [E, H] fp32 -> fp32 logits [b, E]
    (providers page, MoEProvider docstring; RoutedMoE.build: the router reads
    the bf16 MoE input). Exact dot products in float64, stored as fp32."""
    x = bf16_to_f64(x_bf16)
    w = np.asarray(w_router, dtype=np.float64)
    return round_f32(x @ w.T)


@dataclasses.dataclass
class Routing:
    ids: np.ndarray        # int32 [b, k], by descending selection score
    weights: np.ndarray    # fp32 values [b, k]
    scores: np.ndarray     # fp32 values [b, E], unbiased (after sigmoid/softmax)
    selection: np.ndarray  # fp32 values [b, E], scores + bias
    gap: np.ndarray        # [b] selection[k-th] - selection[(k+1)-th]; inf if k == E


def weights_for_ids(scores, ids, route_scale: float, division_eps=None) -> np.ndarray:
    """Gather the UNBIASED scores of the selected ids, divide by (their sum +
    division_eps), multiply by route_scale; stored as fp32 (muse_moe_runner
    page, MuseSpark1xRouter._compute_routing_native, after the top-k)."""
    ids = np.asarray(ids, dtype=np.int64)
    rows = np.arange(ids.shape[0])[:, None]
    w = np.asarray(scores, dtype=np.float64)[rows, ids]
    denom = w.sum(axis=-1, keepdims=True)
    if division_eps is not None:
        denom = denom + float(np.float32(division_eps))
    return round_f32(w / denom * float(np.float32(route_scale)))


def route(logits, expert_bias, top_k: int, route_scale: float,
          multiplier: float | None = None, score: str = "sigmoid",
          division_eps: float | None = None) -> Routing:
    """The MuseSpark1x routing rule (muse_moe_runner page, MuseSpark1xRouter
    docstring and ``_compute_routing_native``):

    optional output multiplier -> sigmoid or softmax -> add the expert bias for
    SELECTION only -> top-k -> gather the UNBIASED scores -> divide by
    (sum + division_eps) -> multiply by route_scale.

    The recipe runs on fp32 tensors, so the multiplied logits, the scores and
    the selection scores are stored as fp32 here too, and the top-k decision
    is taken on fp32 values. Reading: torch.topk's order of equal values is
    not fixed by the page; here equal selection scores go to the lower expert
    id first. The weights are computed in float64 from the fp32 scores and
    stored as fp32 (the recipe's ``.to(torch.float32)``).
    """
    if score not in ("sigmoid", "softmax"):
        raise ValueError(f"Invalid router_score_normalization: {score}")
    g = np.asarray(logits, dtype=np.float64)
    b, E = g.shape
    if not 1 <= top_k <= E:
        raise ValueError("top_k must be in [1, E]")
    if multiplier is not None:
        g = round_f32(g * float(np.float32(multiplier)))
    if score == "sigmoid":
        s = round_f32(1.0 / (1.0 + np.exp(-g)))
    else:
        z = np.exp(g - g.max(axis=-1, keepdims=True))
        s = round_f32(z / z.sum(axis=-1, keepdims=True))
    sel = round_f32(s + np.asarray(expert_bias, dtype=np.float32).astype(np.float64))
    order = np.argsort(-sel, axis=-1, kind="stable")   # ties keep the lower id first
    ids = order[:, :top_k]
    rows = np.arange(b)[:, None]
    if top_k < E:
        gap = sel[rows[:, 0], ids[:, -1]] - sel[rows[:, 0], order[:, top_k]]
    else:
        gap = np.full(b, np.inf)
    weights = weights_for_ids(s, ids, route_scale, division_eps)
    return Routing(ids.astype(np.int32), weights, s, sel, gap)


# --------------------------------------------------------------------------
# Pooler, pre-expert norm, activation quantization
# --------------------------------------------------------------------------


def pre_expert(x_bf16, w_pool_bf16, w_pre_norm_bf16, eps: float,
               pre_norm: bool = True, near=None, ties=None) -> np.ndarray:
    """Pooler GEMM H -> P, then pre_expert_norm (providers page, MoEProvider
    docstring, which lists the pooler GEMM, the gather and pre_expert_norm as
    one stage). The pooled vector
    is not rounded before the norm (the pooler and the norm run fused); the
    result h is stored as bf16 (decoder page, _K5Bucket buffer ``h`` bf16)."""
    h_raw = bf16_to_f64(x_bf16) @ bf16_to_f64(w_pool_bf16).T
    if pre_norm:
        h_raw = rms_norm(h_raw, bf16_to_f64(w_pre_norm_bf16), eps)
    h, n = round_bf16_near(h_raw, near)
    if ties is not None:
        ties["h"] = ties.get("h", 0) + n
    return h


def quantize_rows_e4m3(v: np.ndarray):
    """Per-row dynamic e4m3 quantization of bf16-valued activations:
    scale = fp32(amax / 448), codes = e4m3(fp32(v / scale)) (round to nearest
    even, saturating). A row whose amax is 0 gets scale 0 and zero codes.
    (The pages do not show the FP8 activation quantizer; this is the plain
    per-row dynamic form.)"""
    v = np.asarray(v, dtype=np.float64)
    amax = np.abs(v).max(axis=-1, keepdims=True)
    scale = round_f32(amax / 448.0)
    safe = np.where(scale > 0, scale, 1.0)
    q = np.where(scale > 0, e4m3_encode(round_f32(v / safe)), 0).astype(np.uint8)
    return q, scale[..., 0]


def quantize_act_nvfp4(v: np.ndarray):
    """Dynamic NVFP4 quantization of bf16-valued activations [..., K] into the
    expert input the stock layer hands the routed experts (providers page,
    ExpertsInput: two e2m1 codes per byte, one e4m3 block scale per 16).

    Reading (ExpertsInput carries codes and block scales and no global scale;
    the page prints no quantizer): per block of 16 consecutive elements, the
    scale is the e4m3 value nearest fp32(amax / 6) (ties to even, saturating
    at 448), 6 being the largest e2m1 magnitude; each element becomes the
    e2m1 magnitude nearest fp32(|v| / scale), ties to the even code,
    saturating at 6, with the sign bit of v; a block whose scale is 0 gets
    magnitude 0 everywhere (sign bits kept).

    Returns (codes uint8 [..., K/2], element 2j in the low nibble of byte j;
    scales e4m3 uint8 [..., K/16])."""
    v = np.asarray(v, dtype=np.float64)
    K = v.shape[-1]
    assert K % 16 == 0
    blk = v.reshape(v.shape[:-1] + (K // 16, 16))
    amax = np.abs(blk).max(axis=-1)
    s_code = e4m3_encode(round_f32(amax / 6.0))
    sf = e4m3_decode(s_code)
    safe = np.where(sf > 0, sf, 1.0)[..., None]
    a = np.where(sf[..., None] > 0, round_f32(np.abs(blk) / safe), 0.0)
    # every quotient of 6 or more saturates to 6; bounding it keeps the
    # distances below exact (at quotients near 1e35 they would all be equal)
    a = np.minimum(a, 8.0)
    d = np.abs(a[..., None] - E2M1[:8])
    best = d.min(axis=-1, keepdims=True)
    cand = d == best
    even = cand & ((np.arange(8) & 1) == 0)
    code = np.where(even.any(axis=-1), np.argmax(even, axis=-1), np.argmax(cand, axis=-1))
    code = code.astype(np.uint8) | (np.signbit(blk).astype(np.uint8) << 3)
    codes = code.reshape(v.shape)
    packed = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
    return packed, s_code


def fp4_activation(v: np.ndarray, fmt: str) -> np.ndarray:
    """The values a W4A4 expert GEMM multiplies: bf16-valued activations
    [..., K] rounded to MXFP4 (the OCP rule of quantize_mxfp4; muse_moe_runner
    page, the Quark w_mxfp4_a_mxfp4 scheme with dynamic MXFP4 activations) or
    to NVFP4 (quantize_act_nvfp4), then decoded exactly."""
    v = np.asarray(v, dtype=np.float64)
    K = v.shape[-1]
    if fmt == "mxfp4":
        packed, sc = quantize_mxfp4(f64_to_bf16_bits(v))
        vals = E2M1[unpack_fp4(packed)]
        return (vals.reshape(v.shape[:-1] + (K // 32, 32)) * ue8m0_decode(sc)[..., None]).reshape(v.shape)
    if fmt == "nvfp4":
        packed, sc = quantize_act_nvfp4(v)
        vals = E2M1[unpack_fp4(packed)]
        return (vals.reshape(v.shape[:-1] + (K // 16, 16)) * e4m3_decode(sc)[..., None]).reshape(v.shape)
    raise ValueError(fmt)


# --------------------------------------------------------------------------
# Routed experts
# --------------------------------------------------------------------------


# the two e2m1 values of every byte: low nibble first
_FP4_BYTE_VALUES = np.stack([E2M1[np.arange(256) & 0x0F], E2M1[np.arange(256) >> 4]], axis=-1)


def _fp4_values(packed: np.ndarray) -> np.ndarray:
    """[N, K/2] packed e2m1 bytes -> [N, K] float64 (same order as unpack_fp4)."""
    return _FP4_BYTE_VALUES[packed].reshape(packed.shape[0], -1)


def _apply_block_scale(vals: np.ndarray, scale: np.ndarray, block: int) -> np.ndarray:
    """Multiply [N, K] values by one scale per `block` consecutive K ([N, K/block])."""
    N, K = vals.shape
    return (vals.reshape(N, K // block, block) * scale[:, :, None]).reshape(N, K)


def dequant_expert(quant: str, t: dict, e: int):
    """Expert e's fused w13 [2I, P] and w2 [P, I] as float64 (exact).

    MXFP4: e2m1 * 2^(s-127), one UE8M0 scale per 32 along K (decoder page,
    MonoDims.expert_shapes). NVFP4: e2m1 * e4m3 block scale per 16 along K *
    fp32 global scale of the expert. FP8: e4m3 * fp32 scale per output row.
    BF16: the bf16 values (the unquantized experts of the first and last
    decoder layers: muse_moe_runner page, MuseSparkUnquantizedFusedMoE and
    _online_mxfp4_applies). The W4A4 forms ("mxfp4_a4", "nvfp4_a4") hold
    their weights as MXFP4 / NVFP4.
    """
    quant = {"mxfp4_a4": "mxfp4", "nvfp4_a4": "nvfp4"}.get(quant, quant)
    if quant == "mxfp4":
        w13 = _apply_block_scale(_fp4_values(t["w13"][e]), ue8m0_decode(t["w13_scale"][e]), 32)
        w2 = _apply_block_scale(_fp4_values(t["w2"][e]), ue8m0_decode(t["w2_scale"][e]), 32)
    elif quant == "nvfp4":
        w13 = _apply_block_scale(_fp4_values(t["w13"][e]), e4m3_decode(t["w13_scale"][e]), 16)
        w13 *= float(t["w13_gscale"][e])
        w2 = _apply_block_scale(_fp4_values(t["w2"][e]), e4m3_decode(t["w2_scale"][e]), 16)
        w2 *= float(t["w2_gscale"][e])
    elif quant == "fp8":
        w13 = e4m3_decode(t["w13"][e]) * t["w13_scale"][e].astype(np.float64)[:, None]
        w2 = e4m3_decode(t["w2"][e]) * t["w2_scale"][e].astype(np.float64)[:, None]
    elif quant == "bf16":
        w13 = bf16_to_f64(t["w13"][e])
        w2 = bf16_to_f64(t["w2"][e])
    else:
        raise ValueError(quant)
    return w13, w2


def silu(z):
    return z / (1.0 + np.exp(-z))


def expert_outputs(h: np.ndarray, ids: np.ndarray, quant: str, t: dict,
                   inter: int, act_out: np.ndarray | None = None, near_act=None,
                   ties=None) -> np.ndarray:
    """One unweighted output per selected route, y [b, k, P] (muse_moe_runner
    page, MuseSparkAiterExperts: the experts run with unit weights so that
    the router weighting happens after the post-expert norm).

    Per route (t, j) with e = ids[t, j]: gu = W13_e h_t; gate = gu[:I],
    up = gu[I:] (reading: the vLLM fused-w13 order, gate rows first);
    a = bf16(silu(gate) * up) (the MoE activations are bf16); y = W2_e a.
    FP8 W8A8 quantizes both expert inputs per row (quantize_rows_e4m3) and
    multiplies the e4m3 values back by their scales. W4A4 ("mxfp4_a4",
    "nvfp4_a4") rounds both expert inputs, h per token and a per route, to
    the weights' FP4 format (fp4_activation). ``act_out`` ([b, k, I]),
    when given, receives the bf16 activations; ``near_act`` applies the
    near-tie rule of round_bf16_near to their rounding.
    """
    b, k = ids.shape
    P = h.shape[-1]
    y = np.zeros((b, k, P))
    a4 = {"mxfp4_a4": "mxfp4", "nvfp4_a4": "nvfp4"}.get(quant)
    if quant == "fp8":
        qh, sh = quantize_rows_e4m3(h)
        h_in = e4m3_decode(qh) * sh[:, None]
    elif a4 is not None:
        h_in = fp4_activation(h, a4)
    else:
        h_in = h
    for e in np.unique(ids):
        tok, slot = np.nonzero(ids == e)
        w13, w2 = dequant_expert(quant, t, int(e))
        gu = h_in[tok] @ w13.T                       # [n, 2I]
        a, n = round_bf16_near(silu(gu[:, :inter]) * gu[:, inter:],
                               None if near_act is None else near_act[tok, slot])
        if ties is not None:
            ties["act"] = ties.get("act", 0) + n
        if act_out is not None:
            act_out[tok, slot] = a
        if quant == "fp8":
            qa, sa = quantize_rows_e4m3(a)
            a = e4m3_decode(qa) * sa[:, None]
        elif a4 is not None:
            a = fp4_activation(a, a4)
        y[tok, slot] = a @ w2.T
    return y


# --------------------------------------------------------------------------
# Tail, unpooler, FFN boundary
# --------------------------------------------------------------------------


def finalize(y: np.ndarray, weights: np.ndarray, w_post_bf16, eps: float, near=None,
             ties=None) -> np.ndarray:
    """post_expert_norm of every route row, times its router weight, summed
    over the k routes (muse_moe_runner page, MuseSparkTopKWeightAndReduce.apply,
    unfused branch); the result moe_out is stored as bf16 (providers page,
    RoutedMoE buffer ``moe_out``)."""
    n = rms_norm(y, bf16_to_f64(w_post_bf16), eps)
    out, c = round_bf16_near((n * np.asarray(weights, dtype=np.float64)[..., None]).sum(axis=1),
                             near)
    if ties is not None:
        ties["moe_out"] = ties.get("moe_out", 0) + c
    return out


def unpool(moe_out: np.ndarray, w_unpool_bf16) -> np.ndarray:
    """Unpooler GEMM P -> H (providers page, MoEProvider docstring). Not rounded:
    it feeds the boundary directly."""
    return np.asarray(moe_out, dtype=np.float64) @ bf16_to_f64(w_unpool_bf16).T


def boundary(u: np.ndarray, stream, w_ffn_norm_bf16, gate: float,
             w_next_norm_bf16, eps: float, near=None, ties=None):
    """FFN boundary (providers page, BoundaryProvider docstring): post_ffn_norm
    of u, gated add into the fp32 stream in place, next pre-norm into bf16 out.
    Reading: the gated add is stream + gate * post_ffn_norm(u), one scalar gate
    per layer (the decoder page names add_ffn alpha/beta but not the formula).
    Returns (new stream as fp32 values, out as bf16 values)."""
    add = rms_norm(u, bf16_to_f64(w_ffn_norm_bf16), eps)
    s_new = round_f32(np.asarray(stream, dtype=np.float64) + float(np.float32(gate)) * add)
    out, c = round_bf16_near(rms_norm(s_new, bf16_to_f64(w_next_norm_bf16), eps), near)
    if ties is not None:
        ties["out"] = ties.get("out", 0) + c
    return s_new, out


def attention_boundary(partial_bf16: np.ndarray, stream, gate: float, w_pre_ffn_bf16,
                       eps: float, near=None, ties=None):
    """Attention boundary, the step before the block (providers page,
    AttentionBoundaryProvider docstring): post_attn_norm of the o_proj output
    ``partial`` (bf16), gated add into the fp32 stream in place, pre_ffn_norm
    into bf16 out (the block's input x). post_attn_norm has no weight (decoder
    page: each layer's check rejects a post_attn_norm with a weight). The
    all-reduce of ``partial`` over ranks is outside this one-GPU path:
    ``partial`` is the summed output. Reading, as for the FFN boundary: the
    gated add is stream + gate * post_attn_norm(partial) with one scalar gate.
    Returns (new stream as fp32 values, out as bf16 values)."""
    add = rms_norm(bf16_to_f64(partial_bf16), 1.0, eps)
    s_new = round_f32(np.asarray(stream, dtype=np.float64) + float(np.float32(gate)) * add)
    out, c = round_bf16_near(rms_norm(s_new, bf16_to_f64(w_pre_ffn_bf16), eps), near)
    if ties is not None:
        ties["out"] = ties.get("out", 0) + c
    return s_new, out


# --------------------------------------------------------------------------
# The block
# --------------------------------------------------------------------------


def block(x_bf16, stream, w: dict, *, top_k: int, route_scale: float,
          multiplier=None, score="sigmoid", division_eps=None, quant="mxfp4",
          norm_eps=1e-6, pre_norm=True, force_ids=None, near=None) -> dict:
    """One MoE decode block followed by its FFN boundary.

    ``w`` holds the layer's tensors in storage form (see synth.layer_tensors).
    ``force_ids`` replaces the selected ids (same order) to continue the chain
    on another valid selection at a near tie; the weights are then recomputed
    from those ids with the same rule. ``near`` (dict with any of h, act,
    moe_out, out) applies the near-tie rule of round_bf16_near at those
    rounding points; result["near_ties"] counts the elements it decided.
    Returns every intermediate: logits, routing, h, y, moe_out, u, stream, out
    (and out_bits, the bf16 bit patterns of out).
    """
    logits = router_logits(x_bf16, w["w_router"])
    r = route(logits, w["expert_bias"], top_k, route_scale, multiplier, score, division_eps)
    if force_ids is not None:
        ids = np.asarray(force_ids, dtype=np.int32)
        r = Routing(ids, weights_for_ids(r.scores, ids, route_scale, division_eps),
                    r.scores, r.selection, r.gap)
    near = near or {}
    ties: dict = {}
    h = pre_expert(x_bf16, w["w_pool"], w["w_pre_norm"], norm_eps, pre_norm, near.get("h"), ties)
    inter = (w["w13"].shape[1]) // 2
    act = np.zeros(r.ids.shape + (inter,))
    y = expert_outputs(h, r.ids, quant, w, inter, act, near.get("act"), ties)
    moe_out = finalize(y, r.weights, w["w_post_norm"], norm_eps, near.get("moe_out"), ties)
    u = unpool(moe_out, w["w_unpool"])
    s_new, out = boundary(u, stream, w["w_ffn_norm"], float(w["gate"][0]),
                          w["w_next_norm"], norm_eps, near.get("out"), ties)
    return dict(logits=logits, routing=r, ids=r.ids, weights=r.weights, gap=r.gap,
                h=h, act=act, y=y, moe_out=moe_out, u=u, stream=s_new, out=out,
                out_bits=f64_to_bf16_bits(out), near_ties=ties)
