"""Python binding of libmusemoe (the MuseSpark1x MoE decode block on GB300).

Argument marshalling only: every step of the block runs in the library's CUDA
kernels (``csrc/``, C ABI in ``include/musemoe.h``). The functions carry the
C names. Tensors may be passed as torch tensors (their ``data_ptr()`` is
used) or as raw integer addresses; streams as ``torch.cuda.Stream``, a raw
``cudaStream_t`` integer, or None for torch's current stream.

There is no fallback: if ``libmusemoe.so`` has not been built every call
raises. Build it with ``moe_decode_layer_router_gb300._build.build()``.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

__all__ = [
    "MUSEMOE_OK", "MUSEMOE_EINVAL", "MUSEMOE_EUNSUPPORTED", "MUSEMOE_ECUDA", "MUSEMOE_ENOMEM",
    "MUSEMOE_ERANGE", "MUSEMOE_ETIMEOUT", "MUSEMOE_MXFP4", "MUSEMOE_NVFP4", "MUSEMOE_FP8_W8A8", "MUSEMOE_BF16",
    "MUSEMOE_MXFP4_A4", "MUSEMOE_NVFP4_A4", "MUSEMOE_SIGMOID",
    "MUSEMOE_SOFTMAX", "Dims", "Config", "Weights", "Taps", "MuseMoEError", "library",
    "musemoe_create", "musemoe_destroy", "musemoe_last_error", "musemoe_workspace_bytes",
    "musemoe_num_kernels", "musemoe_kernel_name", "musemoe_pack_experts", "musemoe_route",
    "musemoe_forward", "musemoe_forward_debug", "musemoe_forward_host", "musemoe_poll_health",
    "musemoe_route_static", "musemoe_attention_boundary", "musemoe_quantize_mxfp4",
    "musemoe_quantize_act_nvfp4", "musemoe_health_selftest", "musemoe_set_expert_path",
    "musemoe_forward_ep_partial", "musemoe_forward_ep_combine", "MUSEMOE_PATH_AUTO", "MUSEMOE_PATH_MMA", "MUSEMOE_PATH_TCGEN05", "EXPORTED_SYMBOLS",
    "WEIGHT_FIELDS",
]

(MUSEMOE_OK, MUSEMOE_EINVAL, MUSEMOE_EUNSUPPORTED, MUSEMOE_ECUDA, MUSEMOE_ENOMEM, MUSEMOE_ERANGE,
 MUSEMOE_ETIMEOUT) = (0, 1, 2, 3, 4, 5, 6)
MUSEMOE_MXFP4, MUSEMOE_NVFP4, MUSEMOE_FP8_W8A8, MUSEMOE_BF16 = 0, 1, 2, 3
MUSEMOE_MXFP4_A4, MUSEMOE_NVFP4_A4 = 4, 5
MUSEMOE_SIGMOID, MUSEMOE_SOFTMAX = 0, 1
MUSEMOE_PATH_AUTO, MUSEMOE_PATH_MMA, MUSEMOE_PATH_TCGEN05 = 0, 1, 2
_STATUS = {0: "OK", 1: "EINVAL", 2: "EUNSUPPORTED", 3: "ECUDA", 4: "ENOMEM", 5: "ERANGE",
           6: "ETIMEOUT"}

c_i32, c_f32, c_vp = ctypes.c_int32, ctypes.c_float, ctypes.c_void_p


class Dims(ctypes.Structure):
    _fields_ = [("max_rows", c_i32), ("hidden", c_i32), ("pooled", c_i32), ("inter", c_i32),
                ("experts", c_i32), ("top_k", c_i32)]


class Config(ctypes.Structure):
    _fields_ = [("score", c_i32), ("route_scale", c_f32), ("has_multiplier", c_i32),
                ("multiplier", c_f32), ("has_division_eps", c_i32), ("division_eps", c_f32),
                ("norm_eps", c_f32), ("pre_expert_norm", c_i32)]


WEIGHT_FIELDS = ["w_router", "expert_bias", "w_pool", "w_pre_norm", "w13", "w13_scale",
                 "w13_gscale", "w2", "w2_scale", "w2_gscale", "w_post_norm", "w_unpool",
                 "w_ffn_norm", "w_next_norm", "gate"]


class Weights(ctypes.Structure):
    _fields_ = [(n, c_vp) for n in WEIGHT_FIELDS]


class Taps(ctypes.Structure):
    _fields_ = [("logits", c_vp), ("ids", c_vp), ("weights", c_vp), ("h", c_vp), ("act", c_vp),
                ("y", c_vp), ("moe_out", c_vp), ("u", c_vp), ("events", c_vp)]


EXPORTED_SYMBOLS = [
    "musemoe_create", "musemoe_destroy", "musemoe_last_error", "musemoe_workspace_bytes",
    "musemoe_num_kernels", "musemoe_kernel_name", "musemoe_pack_experts", "musemoe_route",
    "musemoe_forward", "musemoe_forward_debug", "musemoe_forward_host", "musemoe_poll_health",
    "musemoe_route_static", "musemoe_attention_boundary", "musemoe_quantize_mxfp4",
    "musemoe_quantize_act_nvfp4", "musemoe_health_selftest", "musemoe_set_expert_path",
    "musemoe_forward_ep_partial", "musemoe_forward_ep_combine",
]
MUSEMOE_STATIC_MAX_ROWS = 64
MUSEMOE_STATIC_SCRATCH_BYTES = 64 * 1024


class MuseMoEError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"musemoe {_STATUS.get(status, status)}: {message}")
        self.status = status


_lib = None


def library() -> ctypes.CDLL:
    """The loaded libmusemoe.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError(
                f"{_build.LIB} is not built; run moe_decode_layer_router_gb300._build.build()")
        lib = ctypes.CDLL(_build.LIB)
        P = ctypes.POINTER
        lib.musemoe_create.argtypes = [P(Dims), c_i32, P(Config), P(c_vp)]
        lib.musemoe_destroy.argtypes = [c_vp]
        lib.musemoe_destroy.restype = None
        lib.musemoe_last_error.argtypes = [c_vp]
        lib.musemoe_last_error.restype = ctypes.c_char_p
        lib.musemoe_workspace_bytes.argtypes = [P(Dims), c_i32]
        lib.musemoe_workspace_bytes.restype = ctypes.c_size_t
        lib.musemoe_num_kernels.argtypes = [c_i32]
        lib.musemoe_kernel_name.argtypes = [c_i32, c_i32]
        lib.musemoe_kernel_name.restype = ctypes.c_char_p
        lib.musemoe_pack_experts.argtypes = [P(Dims), c_i32] + [c_vp] * 9
        lib.musemoe_route.argtypes = [c_vp, P(Weights), c_vp, c_i32, c_vp, c_vp, c_vp]
        lib.musemoe_forward.argtypes = [c_vp, P(Weights), c_vp, c_vp, c_vp, c_i32, c_vp]
        lib.musemoe_forward_debug.argtypes = [c_vp, P(Weights), c_vp, c_vp, c_vp, c_i32, c_vp,
                                              P(Taps)]
        lib.musemoe_forward_host.argtypes = [c_vp, P(Weights), c_vp, c_vp, c_vp, c_i32, c_vp]
        lib.musemoe_poll_health.argtypes = [c_vp]
        lib.musemoe_route_static.argtypes = [c_i32, c_i32, c_i32, P(Config), c_vp, c_vp, c_vp,
                                             c_i32, c_vp, c_vp, c_vp]
        lib.musemoe_attention_boundary.argtypes = [c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, c_i32,
                                                   c_f32, c_vp]
        lib.musemoe_quantize_mxfp4.argtypes = [c_vp, c_vp, c_vp, ctypes.c_int64, c_i32, c_vp]
        lib.musemoe_quantize_act_nvfp4.argtypes = [c_vp, c_vp, c_vp, ctypes.c_int64, c_i32, c_vp]
        lib.musemoe_health_selftest.argtypes = [c_vp, c_vp]
        lib.musemoe_set_expert_path.argtypes = [c_vp, c_i32]
        lib.musemoe_forward_ep_partial.argtypes = [c_vp, P(Weights), c_vp, c_vp, c_i32, c_i32,
                                                   c_i32, c_vp]
        lib.musemoe_forward_ep_combine.argtypes = [c_vp, P(Weights), c_vp, c_vp, c_vp, c_i32,
                                                   c_vp]
        for name in EXPORTED_SYMBOLS:
            f = getattr(lib, name)
            if f.restype is ctypes.c_int:  # ctypes default
                f.restype = c_i32
        _lib = lib
    return _lib


def _addr(x) -> int | None:
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return int(x)


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    return int(s)


def _check(status: int, handle=None) -> None:
    if status != MUSEMOE_OK:
        raise MuseMoEError(status, musemoe_last_error(handle))


def musemoe_last_error(handle=None) -> str:
    return library().musemoe_last_error(handle).decode()


def musemoe_create(dims: Dims, quant: int, config: Config):
    h = c_vp()
    _check(library().musemoe_create(ctypes.byref(dims), quant, ctypes.byref(config),
                                    ctypes.byref(h)))
    return h


def musemoe_destroy(handle) -> None:
    library().musemoe_destroy(handle)


def musemoe_workspace_bytes(dims: Dims, quant: int) -> int:
    return library().musemoe_workspace_bytes(ctypes.byref(dims), quant)


def musemoe_num_kernels(quant: int) -> int:
    return library().musemoe_num_kernels(quant)


def musemoe_kernel_name(quant: int, i: int) -> str:
    return library().musemoe_kernel_name(quant, i).decode()


def musemoe_pack_experts(dims: Dims, quant: int, w13_src, w13_scale_src, w13_dst, w13_scale_dst,
                         w2_src, w2_scale_src, w2_dst, w2_scale_dst, stream=None) -> None:
    _check(library().musemoe_pack_experts(
        ctypes.byref(dims), quant, _addr(w13_src), _addr(w13_scale_src), _addr(w13_dst),
        _addr(w13_scale_dst), _addr(w2_src), _addr(w2_scale_src), _addr(w2_dst),
        _addr(w2_scale_dst), _stream(stream)))


def musemoe_route(handle, weights: Weights, x, rows: int, ids_out, weights_out,
                  stream=None) -> None:
    _check(library().musemoe_route(handle, ctypes.byref(weights), _addr(x), rows,
                                   _addr(ids_out), _addr(weights_out), _stream(stream)), handle)


def musemoe_forward(handle, weights: Weights, x, stream_io, out, rows: int,
                    stream=None) -> None:
    _check(library().musemoe_forward(handle, ctypes.byref(weights), _addr(x), _addr(stream_io),
                                     _addr(out), rows, _stream(stream)), handle)


def musemoe_forward_debug(handle, weights: Weights, x, stream_io, out, rows: int, stream=None,
                          taps: Taps | None = None) -> None:
    _check(library().musemoe_forward_debug(handle, ctypes.byref(weights), _addr(x),
                                           _addr(stream_io), _addr(out), rows, _stream(stream),
                                           ctypes.byref(taps) if taps is not None else None),
           handle)


def musemoe_forward_host(handle, weights: Weights, x_host, stream_host, out_host, rows: int,
                         stream=None) -> None:
    _check(library().musemoe_forward_host(handle, ctypes.byref(weights), _addr(x_host),
                                          _addr(stream_host), _addr(out_host), rows,
                                          _stream(stream)), handle)


def musemoe_poll_health(handle) -> int:
    """MUSEMOE_OK, MUSEMOE_ERANGE (an expert operand left the fp16 range) or
    MUSEMOE_ETIMEOUT (a bounded wait ran out) since the last poll; other
    failures raise."""
    st = library().musemoe_poll_health(handle)
    if st not in (MUSEMOE_OK, MUSEMOE_ERANGE, MUSEMOE_ETIMEOUT):
        _check(st, handle)
    return st


def musemoe_route_static(hidden: int, experts: int, top_k: int, config: Config, w_router,
                         expert_bias, x, rows: int, ids_out, weights_out, stream=None) -> None:
    """musemoe_route without a handle: the library's fixed static scratch,
    no device allocation (see include/musemoe.h)."""
    _check(library().musemoe_route_static(hidden, experts, top_k, ctypes.byref(config),
                                          _addr(w_router), _addr(expert_bias), _addr(x), rows,
                                          _addr(ids_out), _addr(weights_out), _stream(stream)))


def musemoe_attention_boundary(partial, stream_io, out, w_pre_ffn_norm, gate, rows: int,
                               hidden: int, eps: float, stream=None) -> None:
    """The attention boundary before the block (see include/musemoe.h):
    stream_io += gate * RMSNorm(partial); out = bf16(RMSNorm(stream_io) *
    w_pre_ffn_norm). Device tensors; no handle."""
    _check(library().musemoe_attention_boundary(_addr(partial), _addr(stream_io), _addr(out),
                                                _addr(w_pre_ffn_norm), _addr(gate), rows, hidden,
                                                eps, _stream(stream)))


def musemoe_health_selftest(handle, stream=None) -> None:
    """Runs the library's bounded waits on things nothing completes; the next
    musemoe_poll_health returns MUSEMOE_ETIMEOUT (see include/musemoe.h)."""
    _check(library().musemoe_health_selftest(handle, _stream(stream)), handle)


def musemoe_forward_ep_partial(handle, weights: Weights, x, moe_partial, rows: int,
                               expert_first: int, expert_count: int, stream=None) -> None:
    """The rank's partial moe_out (fp32) of an expert-parallel block: its
    experts [expert_first, expert_first + expert_count) only (see
    include/musemoe.h)."""
    _check(library().musemoe_forward_ep_partial(handle, ctypes.byref(weights), _addr(x),
                                                _addr(moe_partial), rows, expert_first,
                                                expert_count, _stream(stream)), handle)


def musemoe_forward_ep_combine(handle, weights: Weights, moe_sum, stream_io, out, rows: int,
                               stream=None) -> None:
    """bf16(moe_sum), the unpooler and the FFN boundary: the back of an
    expert-parallel block after the all-reduce (see include/musemoe.h)."""
    _check(library().musemoe_forward_ep_combine(handle, ctypes.byref(weights), _addr(moe_sum),
                                                _addr(stream_io), _addr(out), rows,
                                                _stream(stream)), handle)


def musemoe_set_expert_path(handle, path: int) -> None:
    """Selects the routed-expert kernels of the handle's later forwards:
    MUSEMOE_PATH_AUTO, _MMA (warp-level) or _TCGEN05 (tensor cores)."""
    _check(library().musemoe_set_expert_path(handle, path), handle)


def musemoe_quantize_mxfp4(w_bf16, codes, scales, rows: int, cols: int, stream=None) -> None:
    """Online rounding of bf16 weights [rows, cols] to MXFP4 codes
    [rows, cols/2] and UE8M0 scales [rows, cols/32] (see include/musemoe.h)."""
    _check(library().musemoe_quantize_mxfp4(_addr(w_bf16), _addr(codes), _addr(scales), rows,
                                            cols, _stream(stream)))


def musemoe_quantize_act_nvfp4(x_bf16, codes, scales, rows: int, cols: int, stream=None) -> None:
    """The NVFP4 expert input: bf16 activations [rows, cols] to e2m1 codes
    [rows, cols/2] and e4m3 block scales [rows, cols/16] (see
    include/musemoe.h)."""
    _check(library().musemoe_quantize_act_nvfp4(_addr(x_bf16), _addr(codes), _addr(scales), rows,
                                                cols, _stream(stream)))


def make_weights(tensors: dict) -> Weights:
    """A Weights struct from a dict of device tensors (or addresses) keyed by
    WEIGHT_FIELDS; missing keys are NULL. The caller keeps the tensors alive."""
    w = Weights()
    for n in WEIGHT_FIELDS:
        setattr(w, n, _addr(tensors.get(n)))
    return w


def make_taps(logits=None, ids=None, weights=None, h=None, act=None, y=None, moe_out=None,
              u=None, events=None) -> Taps:
    t = Taps()
    for n, v in (("logits", logits), ("ids", ids), ("weights", weights), ("h", h), ("act", act),
                 ("y", y), ("moe_out", moe_out), ("u", u)):
        setattr(t, n, _addr(v))
    if events is not None:
        arr = (c_vp * len(events))(*[e.cuda_event if hasattr(e, "cuda_event") else int(e)
                                     for e in events])
        t._events_keepalive = arr
        t.events = ctypes.cast(arr, c_vp)
    return t
