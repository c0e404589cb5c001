"""Seeded synthetic inputs for the MuseSpark1x MoE decode block.

A module of its own: it draws the block's inputs (activations, residual
stream, router/pooler/unpooler/norm weights and the quantized expert tensors
in their plain storage layout) and holds none of the block's arithmetic.
Both the oracle's tests and the CUDA path's tests and benchmark take their
inputs from here; the two sides share nothing else.

The random draws come from ``synth.c`` (counter-based SplitMix64), compiled
with gcc on first use. Every tensor element is a pure function of
(seed, tensor id, index).

The five workloads (``CONFIGS``) are the block's synthetic configurations:
tiny (correctness), decode (b=8, MXFP4), verify (b=64, NVFP4 with 16 hot
experts), large (b=256, FP8 W8A8) and stack (60 chained layers, b=32, MXFP4).
Any parameter a workload does not state takes the tiny workload's value.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "_synth.so")
_lib = None
_lock = threading.Lock()

MXFP4, NVFP4, FP8, BF16 = "mxfp4", "nvfp4", "fp8", "bf16"
# W4A4: MXFP4 / NVFP4 weights, activations rounded to the same FP4 format
MXFP4_A4, NVFP4_A4 = "mxfp4_a4", "nvfp4_a4"
WEIGHT_FORMAT = {MXFP4_A4: MXFP4, NVFP4_A4: NVFP4}
SIGMOID, SOFTMAX = "sigmoid", "softmax"

# Tensor ids of the counter-based generator.
T_X, T_ROUTER, T_BIAS, T_POOL, T_PRE_NORM = 1, 2, 3, 4, 5
T_W13, T_W13_SCALE, T_W13_G, T_W2, T_W2_SCALE, T_W2_G = 6, 7, 8, 9, 10, 11
T_POST_NORM, T_UNPOOL, T_FFN_NORM, T_NEXT_NORM, T_GATE, T_STREAM, T_HOT = (
    12, 13, 14, 15, 16, 17, 18)
T_PARTIAL, T_PRE_FFN_NORM, T_ATTN_GATE = 19, 20, 21
T_W_BF16 = 22  # bf16 expert weights (online MXFP4 rounding)


def build(force: bool = False) -> str:
    """Compile synth.c into _synth.so next to it (gcc, portable flags)."""
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call([
            "gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fopenmp",
            "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, p = ctypes.c_uint64, ctypes.c_void_p
            d, i32 = ctypes.c_double, ctypes.c_int32
            lib.synth_bytes.argtypes = [u64, u64, p, u64, u64]
            lib.synth_normal_f32.argtypes = [u64, u64, p, u64, u64, d, d]
            lib.synth_normal_bf16.argtypes = [u64, u64, p, u64, u64, d, d]
            lib.synth_uniform_f32.argtypes = [u64, u64, p, u64, u64, d, d]
            lib.synth_int_u8.argtypes = [u64, u64, p, u64, u64, i32, i32, i32]
            lib.synth_e4m3_pow2.argtypes = [u64, u64, p, u64, u64, d, d]
            lib.synth_fp8_rows.argtypes = [u64, u64, p, p, u64, u64, u64, d]
            lib.synth_permutation.argtypes = [u64, u64, p, u64]
            for f in (lib.synth_bytes, lib.synth_normal_f32, lib.synth_normal_bf16,
                      lib.synth_uniform_f32, lib.synth_int_u8, lib.synth_e4m3_pow2,
                      lib.synth_fp8_rows, lib.synth_permutation):
                f.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags.c_contiguous
    return a.ctypes.data


# ---- raw fillers (element i of the tensor lands at out.flat[i - start]) ----

def random_bytes(seed, tensor, shape, start=0):
    out = np.empty(shape, np.uint8)
    _load().synth_bytes(seed, tensor, _ptr(out), start, out.size)
    return out


def normal_f32(seed, tensor, shape, mean=0.0, std=1.0, start=0):
    out = np.empty(shape, np.float32)
    _load().synth_normal_f32(seed, tensor, _ptr(out), start, out.size, mean, std)
    return out


def normal_bf16(seed, tensor, shape, mean=0.0, std=1.0, start=0):
    """bfloat16 values, returned as their uint16 bit patterns."""
    out = np.empty(shape, np.uint16)
    _load().synth_normal_bf16(seed, tensor, _ptr(out), start, out.size, mean, std)
    return out


def uniform_f32(seed, tensor, shape, lo, hi, start=0):
    out = np.empty(shape, np.float32)
    _load().synth_uniform_f32(seed, tensor, _ptr(out), start, out.size, lo, hi)
    return out


def int_u8(seed, tensor, shape, lo, hi, offset, start=0):
    out = np.empty(shape, np.uint8)
    _load().synth_int_u8(seed, tensor, _ptr(out), start, out.size, lo, hi, offset)
    return out


def e4m3_pow2(seed, tensor, shape, lo, hi, start=0):
    out = np.empty(shape, np.uint8)
    _load().synth_e4m3_pow2(seed, tensor, _ptr(out), start, out.size, lo, hi)
    return out


def fp8_rows(seed, tensor, nrows, cols, std, row0=0):
    codes = np.empty((nrows, cols), np.uint8)
    scales = np.empty((nrows,), np.float32)
    _load().synth_fp8_rows(seed, tensor, _ptr(codes), _ptr(scales), row0, nrows,
                           cols, std)
    return codes, scales


def permutation(seed, tensor, n):
    out = np.empty((n,), np.int32)
    _load().synth_permutation(seed, tensor, _ptr(out), n)
    return out


# ---- workloads ----

@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    rows: int
    hidden: int
    pooled: int
    inter: int
    experts: int
    top_k: int
    quant: str
    score: str = SIGMOID
    route_scale: float = 2.5
    multiplier: float | None = 1.0
    division_eps: float | None = 1e-20
    norm_eps: float = 1e-6
    seed: int = 0
    layers: int = 1
    hot_experts: int = 0        # experts whose selection bias is hot_bias
    hot_bias: float = 0.3


_BIG = dict(hidden=5120, pooled=2048, inter=1024, experts=128, top_k=8)

CONFIGS = {
    "tiny": Config("tiny", rows=4, hidden=512, pooled=256, inter=128, experts=16,
                   top_k=2, quant=MXFP4, seed=0),
    "decode": Config("decode", rows=8, quant=MXFP4, multiplier=0.5, seed=1, **_BIG),
    "verify": Config("verify", rows=64, quant=NVFP4, score=SOFTMAX,
                     division_eps=1e-6, hot_experts=16, seed=2, **_BIG),
    "large": Config("large", rows=256, quant=FP8, seed=3, **_BIG),
    "stack": Config("stack", rows=32, quant=MXFP4, seed=4, layers=60, **_BIG),
    # BF16 experts (the first and last decoder layers keep them unquantized)
    "edge_tiny": Config("edge_tiny", rows=4, hidden=512, pooled=256, inter=128, experts=16,
                        top_k=2, quant=BF16, seed=5),
    "edge": Config("edge", rows=8, quant=BF16, multiplier=0.5, seed=6,
                   **{**_BIG, "experts": 32}),
    # W4A4 (FP4 weights and FP4 activations)
    "w4a4_tiny": Config("w4a4_tiny", rows=4, hidden=512, pooled=256, inter=128, experts=16,
                        top_k=2, quant=MXFP4_A4, seed=7),
    "w4a4_nv_tiny": Config("w4a4_nv_tiny", rows=5, hidden=512, pooled=256, inter=128,
                           experts=16, top_k=3, quant=NVFP4_A4, score=SOFTMAX, seed=8),
    "w4a4": Config("w4a4", rows=8, quant=MXFP4_A4, multiplier=0.5, seed=9, **_BIG),
    "w4a4_nv": Config("w4a4_nv", rows=64, quant=NVFP4_A4, score=SOFTMAX, division_eps=1e-6,
                      hot_experts=16, seed=10, **_BIG),
}


def layer_seed(cfg: Config, layer: int) -> int:
    return cfg.seed + layer


def activations(cfg: Config, rows: int | None = None):
    """The block input x (bf16 bits, [b, H]) and residual stream (fp32 [b, H])."""
    b = cfg.rows if rows is None else rows
    x = normal_bf16(cfg.seed, T_X, (b, cfg.hidden))
    stream = normal_f32(cfg.seed, T_STREAM, (b, cfg.hidden))
    return x, stream


def attention_boundary_inputs(cfg: Config, rows: int | None = None, hidden: int | None = None):
    """Inputs of the attention boundary before the block: the o_proj output
    partial (bf16 N(0,1), [b, H]), the residual stream (fp32 N(0,1)), the
    pre_ffn_norm weight (bf16 1+N(0,0.05), [H]) and the gate (fp32 U(0.5,1.5))."""
    b = cfg.rows if rows is None else rows
    H = cfg.hidden if hidden is None else hidden
    return {
        "partial": normal_bf16(cfg.seed, T_PARTIAL, (b, H)),
        "stream": normal_f32(cfg.seed, T_STREAM, (b, H)),
        "w_pre_ffn_norm": normal_bf16(cfg.seed, T_PRE_FFN_NORM, (H,), 1.0, 0.05),
        "gate": uniform_f32(cfg.seed, T_ATTN_GATE, (1,), 0.5, 1.5),
    }


def bf16_expert_weights(cfg: Config, shape, std: float = 0.02, start: int = 0):
    """BF16 expert weights of the given shape (N(0, std)), as the BF16 edge
    layers hold them before any rounding."""
    return normal_bf16(cfg.seed, T_W_BF16, shape, 0.0, std, start=start)


def expert_tensors(cfg: Config, layer: int, e0: int = 0, ne: int | None = None):
    """Experts [e0, e0 + ne) of one layer in their plain storage layout.

    MXFP4: w13 u8 [ne, 2I, P/2] (two e2m1 codes per byte, element 2j in the
    low nibble), w13_scale u8 [ne, 2I, P/32] (UE8M0), likewise w2 [ne, P, I/2]
    and w2_scale [ne, P, I/32].
    NVFP4: the same codes, e4m3 block scales per 16 ([.., P/16], [.., I/16])
    and an fp32 global scale per expert and matrix (w13_gscale, w2_gscale).
    W4A4 (MXFP4_A4, NVFP4_A4): the weights of the FP4 format it names.
    BF16: bf16 N(0, 0.02) weights w13 [ne, 2I, P], w2 [ne, P, I], no scales.
    FP8: e4m3 codes w13 [ne, 2I, P], w2 [ne, P, I], fp32 scale per output
    channel (w13_scale [ne, 2I], w2_scale [ne, P]).
    """
    s = layer_seed(cfg, layer)
    E, P, I = cfg.experts, cfg.pooled, cfg.inter
    ne = E - e0 if ne is None else ne
    out = {}
    wq = WEIGHT_FORMAT.get(cfg.quant, cfg.quant)
    if wq in (MXFP4, NVFP4):
        out["w13"] = random_bytes(s, T_W13, (ne, 2 * I, P // 2), start=e0 * 2 * I * P // 2)
        out["w2"] = random_bytes(s, T_W2, (ne, P, I // 2), start=e0 * P * I // 2)
        if wq == MXFP4:
            out["w13_scale"] = int_u8(s, T_W13_SCALE, (ne, 2 * I, P // 32), -8, -4, 127,
                                      start=e0 * 2 * I * P // 32)
            out["w2_scale"] = int_u8(s, T_W2_SCALE, (ne, P, I // 32), -8, -4, 127,
                                     start=e0 * P * I // 32)
        else:
            out["w13_scale"] = e4m3_pow2(s, T_W13_SCALE, (ne, 2 * I, P // 16), -6.0, -2.0,
                                         start=e0 * 2 * I * P // 16)
            out["w2_scale"] = e4m3_pow2(s, T_W2_SCALE, (ne, P, I // 16), -6.0, -2.0,
                                        start=e0 * P * I // 16)
            out["w13_gscale"] = uniform_f32(s, T_W13_G, (ne,), 0.5, 2.0, start=e0)
            out["w2_gscale"] = uniform_f32(s, T_W2_G, (ne,), 0.5, 2.0, start=e0)
    elif cfg.quant == BF16:
        out["w13"] = normal_bf16(s, T_W13, (ne, 2 * I, P), 0.0, 0.02, start=e0 * 2 * I * P)
        out["w2"] = normal_bf16(s, T_W2, (ne, P, I), 0.0, 0.02, start=e0 * P * I)
    elif cfg.quant == FP8:
        c13, s13 = fp8_rows(s, T_W13, ne * 2 * I, P, 0.05, row0=e0 * 2 * I)
        c2, s2 = fp8_rows(s, T_W2, ne * P, I, 0.05, row0=e0 * P)
        out["w13"], out["w13_scale"] = c13.reshape(ne, 2 * I, P), s13.reshape(ne, 2 * I)
        out["w2"], out["w2_scale"] = c2.reshape(ne, P, I), s2.reshape(ne, P)
    else:
        raise ValueError(cfg.quant)
    return out


def dense_tensors(cfg: Config, layer: int):
    """The layer's router, bias, pooler, unpooler, norm weights and gate."""
    s = layer_seed(cfg, layer)
    E, H, P = cfg.experts, cfg.hidden, cfg.pooled
    bias = uniform_f32(s, T_BIAS, (E,), -0.1, 0.1)
    if cfg.hot_experts:
        hot = permutation(s, T_HOT, E)[: cfg.hot_experts]
        bias[hot] = np.float32(cfg.hot_bias)
    return {
        "w_router": normal_f32(s, T_ROUTER, (E, H), 0.0, 0.02),
        "expert_bias": bias,
        "w_pool": normal_bf16(s, T_POOL, (P, H), 0.0, 0.02),
        "w_pre_norm": normal_bf16(s, T_PRE_NORM, (P,), 1.0, 0.05),
        "w_post_norm": normal_bf16(s, T_POST_NORM, (P,), 1.0, 0.05),
        "w_unpool": normal_bf16(s, T_UNPOOL, (H, P), 0.0, 0.02),
        "w_ffn_norm": normal_bf16(s, T_FFN_NORM, (H,), 1.0, 0.05),
        "w_next_norm": normal_bf16(s, T_NEXT_NORM, (H,), 1.0, 0.05),
        "gate": uniform_f32(s, T_GATE, (1,), 0.5, 1.5),
    }


def layer_tensors(cfg: Config, layer: int = 0):
    """All weights of one layer: dense_tensors + expert_tensors."""
    out = dense_tensors(cfg, layer)
    out.update(expert_tensors(cfg, layer))
    return out


def routing_params(cfg: Config) -> dict:
    return dict(top_k=cfg.top_k, route_scale=cfg.route_scale, multiplier=cfg.multiplier,
                score=cfg.score, division_eps=cfg.division_eps)
