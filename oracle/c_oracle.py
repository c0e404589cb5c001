"""The C oracle (oracle/musemoe_oracle.c) through ctypes: the same block as
musemoe_oracle.block, in plain single-threaded C float64 (no BLAS), and the
same source built with OpenMP for the host's cores.

TEST INFRASTRUCTURE ONLY (tests, __graft_entry__.smoke and the CPU-baseline
and reference legs of bench.py).
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "musemoe_oracle.c")
LIBS = {False: os.path.join(HERE, "_oracle.so"), True: os.path.join(HERE, "_oracle_omp.so")}
QUANT = {"mxfp4": 0, "nvfp4": 1, "fp8": 2, "bf16": 3, "mxfp4_a4": 4, "nvfp4_a4": 5}


def build(force: bool = False) -> None:
    """Compiles the single-threaded and the OpenMP library (gcc, IEEE
    arithmetic: no contraction into fused multiply-adds, no fast-math)."""
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("no C compiler for the oracle")
    for omp, lib in LIBS.items():
        if not force and os.path.exists(lib) and os.path.getmtime(lib) >= os.path.getmtime(SRC):
            continue
        tmp = f"{lib}.{os.getpid()}.tmp"
        cmd = [cc, "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared", SRC, "-o", tmp,
               "-lm"] + (["-fopenmp"] if omp else [])
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"oracle build failed:\n{r.stderr}")
        os.replace(tmp, lib)


class _Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("rows", "hidden", "pooled", "inter", "experts",
                                               "top_k", "quant", "softmax", "has_multiplier",
                                               "has_division_eps", "pre_norm")] + [
        ("route_scale", ctypes.c_float), ("multiplier", ctypes.c_float),
        ("division_eps", ctypes.c_float), ("norm_eps", ctypes.c_double)]


class _Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "w_router", "expert_bias", "w_pool", "w_pre_norm", "w13", "w2", "w13_scale", "w2_scale",
        "w13_gscale", "w2_gscale", "w_post_norm", "w_unpool", "w_ffn_norm", "w_next_norm")] + [
        ("gate", ctypes.c_float)]


_libs: dict = {}


def _lib(omp: bool) -> ctypes.CDLL:
    if omp not in _libs:
        build()
        lib = ctypes.CDLL(LIBS[omp])
        lib.musemoe_oracle_block.argtypes = [ctypes.POINTER(_Config), ctypes.POINTER(_Weights)] + \
            [ctypes.c_void_p] * 8
        lib.musemoe_oracle_route.argtypes = [ctypes.POINTER(_Config)] + [ctypes.c_void_p] * 4
        _libs[omp] = lib
    return _libs[omp]


def _cfg(rows, hidden, pooled, inter, experts, top_k, quant, score, route_scale, multiplier,
         division_eps, norm_eps, pre_norm) -> _Config:
    return _Config(rows=rows, hidden=hidden, pooled=pooled, inter=inter, experts=experts,
                   top_k=top_k, quant=QUANT[quant], softmax=int(score == "softmax"),
                   has_multiplier=int(multiplier is not None),
                   has_division_eps=int(division_eps is not None), pre_norm=int(pre_norm),
                   route_scale=route_scale, multiplier=multiplier or 0.0,
                   division_eps=division_eps or 0.0, norm_eps=norm_eps)


def route(logits, expert_bias, top_k: int, route_scale: float, multiplier=None,
          score: str = "sigmoid", division_eps=None):
    """The routing rule on fp32 logits [b, E]: (ids int32 [b, k], weights fp32 [b, k])."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    b, E = lg.shape
    c = _cfg(b, 0, 0, 0, E, top_k, "mxfp4", score, route_scale, multiplier, division_eps, 0.0, 1)
    bias = np.ascontiguousarray(expert_bias, dtype=np.float32)
    ids = np.empty((b, top_k), np.int32)
    wts = np.empty((b, top_k), np.float32)
    if _lib(False).musemoe_oracle_route(ctypes.byref(c), lg.ctypes.data, bias.ctypes.data,
                                        ids.ctypes.data, wts.ctypes.data):
        raise MemoryError("oracle route")
    return ids, wts


def block(x_bf16, stream, w: dict, *, top_k: int, route_scale: float, multiplier=None,
          score="sigmoid", division_eps=None, quant="mxfp4", norm_eps=1e-6, pre_norm=True,
          omp: bool = False) -> dict:
    """One block with its FFN boundary, as musemoe_oracle.block (storage
    forms in, storage forms out): ids, weights, h (bf16 bits), moe_out (bf16
    bits), stream (fp32), out (bf16 bits). ``omp`` runs the OpenMP build."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    st = np.ascontiguousarray(stream, dtype=np.float32)
    b, H = x.shape
    P = w["w_pool"].shape[0]
    I = w["w13"].shape[1] // 2
    E = w["w_router"].shape[0]
    c = _cfg(b, H, P, I, E, top_k, quant, score, route_scale, multiplier, division_eps, norm_eps,
             pre_norm)
    keep = {k: np.ascontiguousarray(v) for k, v in w.items()}
    ptr = lambda k: keep[k].ctypes.data if k in keep else None
    W = _Weights(**{n: ptr(n) for n in ("w_router", "expert_bias", "w_pool", "w_pre_norm", "w13",
                                        "w2", "w13_scale", "w2_scale", "w13_gscale", "w2_gscale",
                                        "w_post_norm", "w_unpool", "w_ffn_norm", "w_next_norm")},
                 gate=float(np.float32(w["gate"][0])))
    out = dict(ids=np.empty((b, top_k), np.int32), weights=np.empty((b, top_k), np.float32),
               h=np.empty((b, P), np.uint16), moe_out=np.empty((b, P), np.uint16),
               stream=np.empty((b, H), np.float32), out=np.empty((b, H), np.uint16))
    if _lib(omp).musemoe_oracle_block(ctypes.byref(c), ctypes.byref(W), x.ctypes.data,
                                      st.ctypes.data, out["ids"].ctypes.data,
                                      out["weights"].ctypes.data, out["h"].ctypes.data,
                                      out["moe_out"].ctypes.data, out["stream"].ctypes.data,
                                      out["out"].ctypes.data):
        raise MemoryError("oracle block")
    return out
