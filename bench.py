"""Benchmark of the MuseSpark1x MoE decode block on GB300 (one JSON line).

A step is one pass of the whole block (router, routing, pooler + pre-expert
norm, grouped experts, post-expert norm + weighted sum, unpooler, FFN
boundary) over one batch of the decode workload: b=8 rows, H=5120, P=2048,
I=1024, E=128, top-8, MXFP4 experts. Steps rotate over 4 independent
weight sets (about 1.9 GB, far beyond the 129 MB L2) so every step reads its
weights from HBM; one CUDA graph holds the 4 forwards in turn, so a replay
runs 4 steps, chained on the device as consecutive layers' blocks would be.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 (under torchrun) runs N independent replicas, one per GPU (the block
has no cross-GPU step): value = rows of all ranks / max over ranks of the
timed region. --impl reference times the oracle (plain C, float64, one host
core) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-block decode rows/s and achieved HBM GB/s vs roofline per bucket (1×GB300)"
WORKLOAD = "decode"
WEIGHT_SETS = 4

# DRAM traffic of one launch of the dominant kernel, from the ncu capture
# summarized in profiles/ (dram__bytes_read.sum + dram__bytes_write.sum) of
# the decode bucket's w13 (48 active experts), with that launch's
# algorithmic bytes: the bench scales it to its own launches by the ratio
# (the traffic grows with the selected experts' bytes). Valid only for the
# kernel source it was taken on.
NCU_TRAFFIC = {"kernel": "w13", "source_sha1": "9d4e2eb8f37c324d628e9e521305f8430d3c94e0",
               "bytes_per_launch": 107081728 + 2624256, "algorithmic_bytes": 107118592}


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true",
                    help="launch every step's kernels directly instead of replaying a CUDA graph")
    ap.add_argument("--bucket", choices=["decode", "verify", "large", "w4a4", "w4a4_nv"], default=None,
                    help="time one single-layer bucket alone (--steps graph replays, --warmup "
                         "debug forwards) and print its object: a bounded run for profiling")
    return ap.parse_args()


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ------------------------------------------------------------ bytes model

def max_over_ranks(v: float, world: int, device=None) -> float:
    """The largest of the ranks' values (the job ends when its slowest rank
    does). Collective over the default process group when world > 1."""
    if world == 1:
        return float(v)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, rows_per_rank: int, steps: int, seconds: float) -> float:
    """Rows per second of the whole job: every rank runs `steps` steps of
    `rows_per_rank` rows (weak scaling), timed by the slowest rank."""
    return world * rows_per_rank * steps / seconds


def algorithmic_bytes(cfg, ids_list):
    """Minimal HBM bytes per kernel and per step: every weight byte the step
    needs once (only the selected experts' codes and scales), every input
    read once and every output written once, at their storage widths."""
    import numpy as np
    b, H, P, I, E, k = cfg.rows, cfg.hidden, cfg.pooled, cfg.inter, cfg.experts, cfg.top_k
    w13_e = 2 * I * P // 2 + 2 * I * P // 32
    w2_e = P * I // 2 + P * I // 32
    routes = b * k
    per = []
    for ids in ids_list:
        active = len(np.unique(ids))
        per.append({
            "router": E * H * 4 + b * H * 2 + b * E * 4 + b * E * 4 + E * 4 + routes * 12,
            "pool": P * H * 2 + b * H * 2 + b * P * 4 + P * 2 + 2 * b * P * 2,
            "w13": active * w13_e + b * P * 2 + routes * I * 2,
            "w2": active * w2_e + routes * I * 2 + routes * P * 4,
            "finalize": routes * P * 4 + routes * 4 + P * 2 + b * P * 2,
            "unpool": H * P * 2 + b * P * 2 + b * H * 4,
            "boundary": b * H * 4 + 2 * b * H * 4 + 2 * H * 2 + b * H * 2,
            "active_experts": active,
            "expert_bytes": active * (w13_e + w2_e),
        })
    return per


# ------------------------------------------------------------ clocks

class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons of one GPU."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            if self.uuid and self.uuid not in parts[0]:
                continue
            rows.append(parts)
        if not rows:
            return None
        mhz = [float(r[1]) for r in rows if r[1].replace(".", "", 1).isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "", 1).isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if "Active" in r[5 + i]
                          and "Not" not in r[5 + i]})
        return {"sm_mhz": statistics.median(mhz) if mhz else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------ oracle leg

ORACLE_SNIPPET = r"""
import json, os, sys, time
sys.path.insert(0, {root!r})
import synth
from oracle import c_oracle as C
cfg = synth.CONFIGS[{workload!r}]
w = synth.layer_tensors(cfg, {layer})
x, st = synth.activations(cfg)
rows = {rows} or cfg.rows
x, st = x[:rows].copy(), st[:rows].copy()
p = synth.routing_params(cfg)
times = []
deadline = time.perf_counter() + {budget}
for i in range({steps}):
    t0 = time.perf_counter()
    C.block(x, st, w, quant=cfg.quant, norm_eps=cfg.norm_eps, omp={omp}, **p)
    times.append(time.perf_counter() - t0)
    if time.perf_counter() > deadline:
        break
print(json.dumps({{"times": times, "rows": rows}}))
"""


def run_oracle(steps: int, budget_s: float, threads: int = 1, workload: str = WORKLOAD,
               rows: int = 0, layer: int = 0) -> dict:
    """Times the C oracle (plain C, float64, no BLAS) on `steps` blocks of
    `workload` (its first `rows` rows, all if 0; layer `layer` of a stack) in
    a child process: the single-threaded build for threads == 1, else the
    OpenMP build of the same source on `threads` threads."""
    from oracle import c_oracle
    c_oracle.build()
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = str(threads)
    code = ORACLE_SNIPPET.format(root=ROOT, workload=workload, steps=steps, budget=budget_s,
                                 rows=rows, layer=layer, omp=threads > 1)
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         check=True)
    return json.loads(out.stdout.strip().splitlines()[-1])


def _hbm_peak():
    """The measured HBM copy bandwidth (GB/s) and its source; the profiling
    recipe's fallback when no measurement is on disk."""
    pk_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peaks = json.load(open(pk_path)) if os.path.exists(pk_path) else {}
    if peaks.get("hbm_gbs"):
        return float(peaks["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _pct(v, q):
    """q-th percentile of the list v (linear interpolation)."""
    import numpy as np
    return float(np.percentile(np.asarray(v, dtype=np.float64), q))


def _stats(us):
    return {"p10_us": _pct(us, 10), "p50_us": _pct(us, 50), "p90_us": _pct(us, 90),
            "mean_us": float(sum(us) / len(us)), "replays": len(us)}


# ------------------------------------------------------------ our arm

def _bench_form(dev, cfg, quant_code: int, steps: int = 200, reps: int = 20,
                flush: bool = False) -> dict:
    """One weight set of ``cfg`` in the form ``quant_code``: the step time of a
    graph of one forward (``steps`` replays after 10), the per-kernel event
    times of ``reps`` debug forwards, and the selected experts. ``flush``
    (for weights that fit in L2): every replay and debug forward is timed
    alone after a 256 MB write that evicts L2."""
    import numpy as np
    import torch

    import moe_decode_layer_router_gb300 as mm
    import synth

    dims = mm.Dims(max_rows=cfg.rows, hidden=cfg.hidden, pooled=cfg.pooled, inter=cfg.inter,
                   experts=cfg.experts, top_k=cfg.top_k)
    conf = mm.Config(score=mm.MUSEMOE_SIGMOID if cfg.score == synth.SIGMOID else mm.MUSEMOE_SOFTMAX,
                     route_scale=cfg.route_scale, has_multiplier=cfg.multiplier is not None,
                     multiplier=cfg.multiplier or 1.0, has_division_eps=cfg.division_eps is not None,
                     division_eps=cfg.division_eps or 0.0, norm_eps=cfg.norm_eps, pre_expert_norm=1)
    handle = mm.musemoe_create(dims, quant_code, conf)

    def to_dev(a):
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    t = {k: to_dev(v) for k, v in synth.layer_tensors(cfg).items()}
    mm.musemoe_pack_experts(dims, quant_code, t["w13"], t.get("w13_scale"), t["w13"],
                            t.get("w13_scale"), t["w2"], t.get("w2_scale"), t["w2"],
                            t.get("w2_scale"))
    w = mm.make_weights(t)
    x, st = synth.activations(cfg)
    xd, sd = to_dev(x), to_dev(st)
    out = torch.empty((cfg.rows, cfg.hidden), dtype=torch.int16, device=dev)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        mm.musemoe_forward(handle, w, xd, sd, out, cfg.rows, s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        mm.musemoe_forward(handle, w, xd, sd, out, cfg.rows, s)
    scrub = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev) if flush else None
    per = []
    with torch.cuda.stream(s):
        for _ in range(10):
            g.replay()
        if flush:
            for _ in range(steps):
                scrub.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(s)
                g.replay()
                e1.record(s)
                e1.synchronize()
                per.append(e0.elapsed_time(e1) * 1e3)
            us = sum(per) / len(per)
        else:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            for _ in range(steps):
                g.replay()
            e1.record(s)
    torch.cuda.synchronize()
    if not flush:
        us = e0.elapsed_time(e1) * 1e3 / steps
    n = mm.musemoe_num_kernels(quant_code)
    names = [mm.musemoe_kernel_name(quant_code, i) for i in range(n)]
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n)]
    for e in ev:  # torch creates an event on its first record
        e.record(s)
    ids = torch.empty((cfg.rows, cfg.top_k), dtype=torch.int32, device=dev)
    dur = {nm: 0.0 for nm in names}
    with torch.cuda.stream(s):
        for _ in range(reps):
            if flush:
                scrub.zero_()
            mm.musemoe_forward_debug(handle, w, xd, sd, out, cfg.rows, s,
                                     mm.make_taps(events=ev, ids=ids))
            s.synchronize()
            for i, nm in enumerate(names):
                dur[nm] += ev[2 * i].elapsed_time(ev[2 * i + 1]) * 1e3 / reps
    active = len(np.unique(ids.cpu().numpy()))
    health = mm.musemoe_poll_health(handle)
    mm.musemoe_destroy(handle)
    del t, g, scrub
    torch.cuda.empty_cache()
    return {"us_per_step": us, "kernel_us": dur, "active_experts": active,
            "replay_stats": _stats(per) if per else None,
            "health": "ok" if health == mm.MUSEMOE_OK else "fp16 range"}


def bench_bf16_experts(dev, hbm_peak: float) -> dict:
    """The decode workload's shapes with BF16 experts (the unquantized form of
    the first and last decoder layers): one weight set of 128 experts (1.6 GB;
    the ~46 experts a step selects, about 560 MB, dwarf L2). Step time of a
    graph of the forward, and the expert phase (w13 + w2 event times) against
    its algorithmic bytes."""
    import dataclasses

    import moe_decode_layer_router_gb300 as mm
    import synth

    cfg = dataclasses.replace(synth.CONFIGS["edge"], experts=128)
    r = _bench_form(dev, cfg, mm.MUSEMOE_BF16)
    us, dur = r["us_per_step"], r["kernel_us"]
    ebytes = r["active_experts"] * (2 * cfg.inter * cfg.pooled + cfg.pooled * cfg.inter) * 2
    e_us = dur["w13"] + dur["w2"]
    return {"workload": f"decode shapes (b={cfg.rows}, H={cfg.hidden}, P={cfg.pooled}, "
                        f"I={cfg.inter}, E={cfg.experts}, top-{cfg.top_k}) with BF16 experts",
            "rows_per_s": cfg.rows / (us / 1e6), "us_per_step": us,
            "active_experts": r["active_experts"], "expert_bytes": ebytes,
            "expert_phase_us": e_us, "expert_phase_gbs": ebytes / (e_us / 1e6) / 1e9,
            "expert_phase_frac": ebytes / (e_us / 1e6) / 1e9 / hbm_peak,
            "kernel_us": dur, "health": r["health"]}


def expert_bytes_per_expert(cfg) -> int:
    """Codes and scales of one expert's w13 and w2 in the workload's form."""
    import synth
    P, I = cfg.pooled, cfg.inter
    q = synth.WEIGHT_FORMAT.get(cfg.quant, cfg.quant)
    if q == synth.MXFP4:
        return 2 * I * P // 2 + 2 * I * P // 32 + P * I // 2 + P * I // 32
    if q == synth.NVFP4:
        return 2 * I * P // 2 + 2 * I * P // 16 + P * I // 2 + P * I // 16 + 8
    if q == synth.FP8:
        return 2 * I * P + 2 * I * 4 + P * I + P * 4
    return (2 * I * P + P * I) * 2  # BF16


def block_bytes(cfg, active: float) -> float:
    """Algorithmic bytes of one forward: the dense weights once, the selected
    experts' codes and scales once, the activations (x, stream in and out,
    out) once."""
    H, P, E = cfg.hidden, cfg.pooled, cfg.experts
    dense = E * H * 4 + E * 4 + 2 * P * H * 2 + (P + 3 * H) * 2
    return dense + active * expert_bytes_per_expert(cfg) + 12 * cfg.rows * H


def block_flops(cfg) -> float:
    """2 x multiply-adds of one forward (router, pooler, routed experts, unpooler)."""
    b, H, P, I, E, k = cfg.rows, cfg.hidden, cfg.pooled, cfg.inter, cfg.experts, cfg.top_k
    return 2.0 * (b * E * H + b * P * H + b * k * (2 * I * P + P * I) + b * H * P)


def bench_bucket(dev, name: str, quant_code: int, hbm_peak: float, cpu_rows: int,
                 cpu_budget: float, replays: int = 200, reps: int = 10) -> dict:
    """One single-layer bucket (a graph of one forward, L2 evicted before each
    replay, 200 replays timed one by one): rows/s at the median, p10/p90, the
    expert phase (w13 + w2 event times) and the whole block against their
    algorithmic bytes, and the oracle on a bounded sample of the same
    workload on one host core."""
    import moe_decode_layer_router_gb300 as mm
    import synth

    cfg = synth.CONFIGS[name]
    r = _bench_form(dev, cfg, quant_code, steps=replays, reps=reps, flush=True)
    st, dur = r["replay_stats"], r["kernel_us"]
    us = st["p50_us"]
    A = r["active_experts"]
    ebytes = A * expert_bytes_per_expert(cfg)
    e_us = dur["w13"] + dur["w2"]
    bbytes = block_bytes(cfg, A)
    eflops = 2.0 * cfg.rows * cfg.top_k * 3 * cfg.inter * cfg.pooled
    cpu = None
    if cpu_rows:
        ora = run_oracle(steps=3, budget_s=cpu_budget, threads=1, workload=name, rows=cpu_rows)
        ot = sum(ora["times"]) / len(ora["times"])
        cpu = {"value": ora["rows"] / ot, "unit": "rows/s", "cores": 1, "kind": "oracle",
               "sample": f"{len(ora['times'])} blocks of the first {ora['rows']} rows "
                         f"({sum(ora['times']):.1f} s, plain C float64, one thread)"}
    return {"workload": f"{name} (b={cfg.rows}, H={cfg.hidden}, P={cfg.pooled}, I={cfg.inter}, "
                        f"E={cfg.experts}, top-{cfg.top_k}, {cfg.quant}, "
                        f"{'softmax' if cfg.score == synth.SOFTMAX else 'sigmoid'}"
                        + (f", {cfg.hot_experts} hot experts" if cfg.hot_experts else "") + ")",
            "timing": "graph of one forward, L2 evicted before each replay", "replays": st,
            "rows_per_s": cfg.rows / (us / 1e6), "us_per_step": us, "active_experts": A,
            "roofline": {"bound": "hbm", "kernel": "w13+w2 (expert phase)", "unit": "GB/s",
                         "algorithmic_bytes": ebytes,
                         "achieved": ebytes / (e_us / 1e6) / 1e9, "peak": hbm_peak,
                         "frac": ebytes / (e_us / 1e6) / 1e9 / hbm_peak},
            "expert_phase_us": e_us,
            "expert_tflops": eflops / (e_us / 1e6) / 1e12,
            "block": {"algorithmic_bytes": bbytes, "achieved_gbs": bbytes / (us / 1e6) / 1e9,
                      "frac": bbytes / (us / 1e6) / 1e9 / hbm_peak,
                      "tflops": block_flops(cfg) / (us / 1e6) / 1e12},
            "kernel_us": dur, "health": r["health"], "cpu_baseline": cpu}


def bench_stack(dev, hbm_peak: float) -> dict:
    """The 60-layer stack (b=32, MXFP4, independent weights per layer, 28 GB,
    far beyond L2): one CUDA graph of the 60 chained forwards (each layer's
    output is the next one's input, the stream carried in place), replayed and
    timed; per layer rows/s, the expert phase of three layers from their
    per-kernel event times, and the oracle on one layer on one host core."""
    import numpy as np
    import torch

    import moe_decode_layer_router_gb300 as mm
    import synth

    cfg = synth.CONFIGS["stack"]
    dims = mm.Dims(max_rows=cfg.rows, hidden=cfg.hidden, pooled=cfg.pooled, inter=cfg.inter,
                   experts=cfg.experts, top_k=cfg.top_k)
    conf = mm.Config(score=mm.MUSEMOE_SIGMOID, route_scale=cfg.route_scale,
                     has_multiplier=int(cfg.multiplier is not None),
                     multiplier=cfg.multiplier or 1.0,
                     has_division_eps=int(cfg.division_eps is not None),
                     division_eps=cfg.division_eps or 0.0, norm_eps=cfg.norm_eps,
                     pre_expert_norm=1)
    handle = mm.musemoe_create(dims, mm.MUSEMOE_MXFP4, conf)

    def to_dev(a):
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    layers = []
    for layer in range(cfg.layers):
        t = {k: to_dev(v) for k, v in synth.layer_tensors(cfg, layer).items()}
        mm.musemoe_pack_experts(dims, mm.MUSEMOE_MXFP4, t["w13"], t["w13_scale"], t["w13"],
                                t["w13_scale"], t["w2"], t["w2_scale"], t["w2"], t["w2_scale"])
        layers.append({"t": t, "w": mm.make_weights(t)})
    x, st = synth.activations(cfg)
    bufs = [to_dev(x), torch.empty_like(to_dev(x))]
    sd = to_dev(st)
    s = torch.cuda.Stream()

    def chain():
        for l_, L in enumerate(layers):
            mm.musemoe_forward(handle, L["w"], bufs[l_ % 2], sd, bufs[(l_ + 1) % 2], cfg.rows, s)

    with torch.cuda.stream(s):
        chain()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        chain()
    per = []
    with torch.cuda.stream(s):
        for _ in range(3):
            g.replay()
        for _ in range(20):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            g.replay()
            e1.record(s)
            e1.synchronize()
            per.append(e0.elapsed_time(e1) * 1e3)
    torch.cuda.synchronize()
    st_ = _stats(per)
    us_layer = st_["p50_us"] / cfg.layers
    # expert phase of three layers (each kernel timed alone)
    n = mm.musemoe_num_kernels(mm.MUSEMOE_MXFP4)
    names = [mm.musemoe_kernel_name(mm.MUSEMOE_MXFP4, i) for i in range(n)]
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n)]
    for e in ev:
        e.record(s)
    ids = torch.empty((cfg.rows, cfg.top_k), dtype=torch.int32, device=dev)
    ebytes, e_us, kern = 0.0, 0.0, {nm: 0.0 for nm in names}
    probe = [0, cfg.layers // 2, cfg.layers - 1]
    with torch.cuda.stream(s):
        for l_ in probe:
            mm.musemoe_forward_debug(handle, layers[l_]["w"], bufs[0], sd, bufs[1], cfg.rows, s,
                                     mm.make_taps(events=ev, ids=ids))
            s.synchronize()
            d = {nm: ev[2 * i].elapsed_time(ev[2 * i + 1]) * 1e3 for i, nm in enumerate(names)}
            for nm in names:
                kern[nm] += d[nm] / len(probe)
            e_us += d["w13"] + d["w2"]
            ebytes += len(np.unique(ids.cpu().numpy())) * expert_bytes_per_expert(cfg)
    health = mm.musemoe_poll_health(handle)
    mm.musemoe_destroy(handle)
    del layers, g
    torch.cuda.empty_cache()
    active = ebytes / len(probe) / expert_bytes_per_expert(cfg)
    bbytes = block_bytes(cfg, active)
    ora = run_oracle(steps=2, budget_s=20.0, threads=1, workload="stack", rows=8, layer=0)
    ot = sum(ora["times"]) / len(ora["times"])
    return {"workload": f"stack ({cfg.layers} chained layers, b={cfg.rows}, H={cfg.hidden}, "
                        f"P={cfg.pooled}, I={cfg.inter}, E={cfg.experts}, top-{cfg.top_k}, "
                        "MXFP4, independent weights per layer)",
            "timing": "one graph of the 60 chained forwards (28 GB of weights, beyond L2)",
            "replays": st_, "us_per_stack": st_["p50_us"], "us_per_layer": us_layer,
            "rows_layers_per_s": cfg.rows * cfg.layers / (st_["p50_us"] / 1e6),
            "active_experts": active,
            "roofline": {"bound": "hbm", "kernel": "w13+w2 (expert phase, 3 layers)",
                         "unit": "GB/s", "algorithmic_bytes": ebytes / len(probe),
                         "achieved": ebytes / (e_us / 1e6) / 1e9, "peak": hbm_peak,
                         "frac": ebytes / (e_us / 1e6) / 1e9 / hbm_peak},
            "block": {"algorithmic_bytes_per_layer": bbytes,
                      "achieved_gbs": bbytes / (us_layer / 1e6) / 1e9,
                      "frac": bbytes / (us_layer / 1e6) / 1e9 / hbm_peak},
            "kernel_us": kern, "health": "ok" if health == mm.MUSEMOE_OK else "fp16 range",
            "cpu_baseline": {"value": ora["rows"] / ot, "unit": "rows*layers/s", "cores": 1,
                             "kind": "oracle",
                             "sample": f"{len(ora['times'])} blocks of layer 0 on "
                                       f"{ora['rows']} rows ({sum(ora['times']):.1f} s, plain "
                                       "C float64, one thread)"}}


def bench_w4a4(dev) -> dict:
    """The decode workload (b=8, E=128, top-8) in the W4A4 forms next to its
    W4A16 form, each timed the same way (one weight set, a graph of one
    forward): what rounding both expert inputs to FP4 costs per step."""
    import dataclasses

    import moe_decode_layer_router_gb300 as mm
    import synth

    res = {"workload": "decode (b=8, H=5120, P=2048, I=1024, E=128, top-8), one weight set, "
                       "graph of one forward"}
    for name, quant, code in [("mxfp4_w4a16", synth.MXFP4, mm.MUSEMOE_MXFP4),
                              ("mxfp4_w4a4", synth.MXFP4_A4, mm.MUSEMOE_MXFP4_A4),
                              ("nvfp4_w4a4", synth.NVFP4_A4, mm.MUSEMOE_NVFP4_A4)]:
        cfg = dataclasses.replace(synth.CONFIGS["decode"], quant=quant)
        r = _bench_form(dev, cfg, code)
        res[name] = {"us_per_step": r["us_per_step"], "rows_per_s": cfg.rows / (r["us_per_step"] / 1e6),
                     "kernel_us": r["kernel_us"], "health": r["health"]}
    return res


def bench_ours(args):
    import numpy as np
    import torch

    import moe_decode_layer_router_gb300 as mm
    import synth
    from moe_decode_layer_router_gb300 import _build

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    _build.build()
    synth.build()
    if args.bucket:
        code = {"decode": mm.MUSEMOE_MXFP4, "verify": mm.MUSEMOE_NVFP4, "large": mm.MUSEMOE_FP8_W8A8,
                "w4a4": mm.MUSEMOE_MXFP4_A4, "w4a4_nv": mm.MUSEMOE_NVFP4_A4}[args.bucket]
        peak, _ = _hbm_peak()
        b = bench_bucket(dev, args.bucket, code, peak, 0 if args.no_cpu_baseline else 16, 15.0,
                         replays=max(1, args.steps), reps=max(3, args.warmup))
        if rank == 0:
            print(json.dumps({"bucket": args.bucket, **b}))
        return
    cfg = synth.CONFIGS[WORKLOAD]
    quant = mm.MUSEMOE_MXFP4
    dims = mm.Dims(max_rows=cfg.rows, hidden=cfg.hidden, pooled=cfg.pooled, inter=cfg.inter,
                   experts=cfg.experts, top_k=cfg.top_k)
    conf = mm.Config(score=mm.MUSEMOE_SIGMOID, route_scale=cfg.route_scale, has_multiplier=1,
                     multiplier=cfg.multiplier, has_division_eps=1,
                     division_eps=cfg.division_eps, norm_eps=cfg.norm_eps, pre_expert_norm=1)
    handle = mm.musemoe_create(dims, quant, conf)

    def to_dev(a):
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    # independent weight sets (different seeds: different weights and routes)
    sets = []
    for r in range(WEIGHT_SETS):
        c = synth.Config(**{**cfg.__dict__, "seed": cfg.seed + 1000 * (r + 1) + 97 * rank})
        t = {k: to_dev(v) for k, v in synth.layer_tensors(c).items()}
        mm.musemoe_pack_experts(dims, quant, t["w13"], t["w13_scale"], t["w13"], t["w13_scale"],
                                t["w2"], t["w2_scale"], t["w2"], t["w2_scale"])
        x, st = synth.activations(c)
        sets.append({"t": t, "w": mm.make_weights(t), "x": to_dev(x), "stream": to_dev(st),
                     "out": torch.empty((cfg.rows, cfg.hidden), dtype=torch.int16, device=dev),
                     "x_host": torch.from_numpy(x.view(np.int16).copy()).pin_memory(),
                     "stream_host": torch.from_numpy(st.copy()).pin_memory()})
    torch.cuda.synchronize()
    set_bytes = sum(v.numel() * v.element_size() for v in sets[0]["t"].values())

    # CUDA graph per set
    s = torch.cuda.Stream()
    graphs = []
    with torch.cuda.stream(s):
        for st_ in sets:
            mm.musemoe_forward(handle, st_["w"], st_["x"], st_["stream"], st_["out"], cfg.rows, s)
    torch.cuda.synchronize()
    for st_ in sets:
        if args.eager:
            def step(st_=st_):
                mm.musemoe_forward(handle, st_["w"], st_["x"], st_["stream"], st_["out"], cfg.rows, s)
            graphs.append(step)
            continue
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            mm.musemoe_forward(handle, st_["w"], st_["x"], st_["stream"], st_["out"], cfg.rows, s)
        graphs.append(g.replay)
    # one graph of the WEIGHT_SETS forwards in turn: a replay runs that many
    # steps, the launches of consecutive forwards chain on the device and
    # the host issues one replay per WEIGHT_SETS steps
    if args.eager:
        def group():
            for f in graphs:
                f()
    else:
        gg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gg, stream=s):
            for st_ in sets:
                mm.musemoe_forward(handle, st_["w"], st_["x"], st_["stream"], st_["out"], cfg.rows, s)
        group = gg.replay
    torch.cuda.synchronize()

    def run_steps(count):
        """count forwards, set i % WEIGHT_SETS for the i-th"""
        i = 0
        while i < count:
            if count - i >= WEIGHT_SETS:
                group()
                i += WEIGHT_SETS
            else:
                graphs[i % WEIGHT_SETS]()
                i += 1

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # warm-up (>= 3 steps)
    with torch.cuda.stream(s):
        run_steps(max(3, args.warmup))
    torch.cuda.synchronize()

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid) if rank == 0 else None
    barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.6)  # the sampler's first reading lands inside the timed region
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        e0.record(s)
        run_steps(args.steps)
        e1.record(s)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    barrier()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    # the step's spread: 200 replays of the graph (WEIGHT_SETS steps each)
    # timed one by one, per step
    rep_us = []
    if not args.eager:
        with torch.cuda.stream(s):
            for _ in range(200):
                r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                r0.record(s)
                group()
                r1.record(s)
                r1.synchronize()
                rep_us.append(r0.elapsed_time(r1) * 1e3 / WEIGHT_SETS)
    kernels = mm.musemoe_num_kernels(quant)
    ms_step = ms / args.steps
    value = whole_job_rate(world, cfg.rows, args.steps, ms / 1e3)

    # per-kernel durations (each kernel timed alone with events) and the
    # selected experts of each set, for the bytes model
    n = kernels
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n)]
    for e in ev:
        e.record(s)
    taps_ids = [torch.empty((cfg.rows, cfg.top_k), dtype=torch.int32, device=dev)
                for _ in sets]
    reps = 50
    dur = [[0.0] * n for _ in sets]
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for rep in range(reps):
            for si, st_ in enumerate(sets):
                tp = mm.make_taps(events=ev, ids=taps_ids[si])
                mm.musemoe_forward_debug(handle, st_["w"], st_["x"], st_["stream"], st_["out"],
                                         cfg.rows, s, tp)
                s.synchronize()
                for i in range(n):
                    dur[si][i] += ev[2 * i].elapsed_time(ev[2 * i + 1]) / reps
    names = [mm.musemoe_kernel_name(quant, i) for i in range(n)]
    ids_np = [t.cpu().numpy() for t in taps_ids]
    model = algorithmic_bytes(cfg, ids_np)
    kernel_ms = {nm: sum(dur[si][i] for si in range(len(sets))) / len(sets)
                 for i, nm in enumerate(names)}
    kernel_bytes = {nm: sum(m[nm] for m in model) / len(model) for nm in names}
    share = {nm: kernel_ms[nm] / sum(kernel_ms.values()) for nm in names}
    dom = max(names, key=lambda nm: kernel_ms[nm])
    hbm_peak, peak_src = _hbm_peak()
    achieved = kernel_bytes[dom] / (kernel_ms[dom] / 1e3) / 1e9
    src = open(os.path.join(ROOT, "moe_decode_layer_router_gb300", "csrc", "k_experts.cu"),
               "rb").read()
    traffic = None
    if (NCU_TRAFFIC["kernel"] == dom and NCU_TRAFFIC["source_sha1"] ==
            hashlib.sha1(src).hexdigest()):
        traffic = (NCU_TRAFFIC["bytes_per_launch"] / NCU_TRAFFIC["algorithmic_bytes"] *
                   kernel_bytes[dom])
    step_bytes = sum(sum(m[nm] for nm in names) for m in model) / len(model)
    expert_bytes = sum(m["expert_bytes"] for m in model) / len(model)
    expert_ms = kernel_ms["w13"] + kernel_ms["w2"]

    # the attention boundary before the block (a separate entry point, not
    # part of the step above): one launch on the workload's rows, timed alone
    ab = synth.attention_boundary_inputs(cfg)
    ab_t = {k: to_dev(v) for k, v in ab.items()}
    ab_out = torch.empty((cfg.rows, cfg.hidden), dtype=torch.int16, device=dev)
    ab_reps = 200
    with torch.cuda.stream(s):
        for _ in range(10):
            mm.musemoe_attention_boundary(ab_t["partial"], ab_t["stream"], ab_out,
                                          ab_t["w_pre_ffn_norm"], ab_t["gate"], cfg.rows,
                                          cfg.hidden, cfg.norm_eps, s)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(s)
        for _ in range(ab_reps):
            mm.musemoe_attention_boundary(ab_t["partial"], ab_t["stream"], ab_out,
                                          ab_t["w_pre_ffn_norm"], ab_t["gate"], cfg.rows,
                                          cfg.hidden, cfg.norm_eps, s)
        a1.record(s)
    torch.cuda.synchronize()
    ab_us = a0.elapsed_time(a1) * 1e3 / ab_reps
    ab_bytes = 12 * cfg.rows * cfg.hidden + 2 * cfg.hidden
    attn_boundary = {"us_per_launch": ab_us, "algorithmic_bytes": ab_bytes,
                     "achieved_gbs": ab_bytes / (ab_us / 1e6) / 1e9,
                     "frac": ab_bytes / (ab_us / 1e6) / 1e9 / hbm_peak,
                     "note": f"{ab_reps} back-to-back launches on the same 0.5 MB (L2-warm); "
                             "latency-bound"}

    # online MXFP4 rounding of bf16 expert weights (load time, not part of
    # the step): w13 of 32 experts, [32 * 2I, P] bf16 = 256 MB (> L2)
    q_rows, q_cols = 32 * 2 * cfg.inter, cfg.pooled
    q_w = to_dev(synth.bf16_expert_weights(cfg, (q_rows, q_cols)))
    q_codes = torch.empty((q_rows, q_cols // 2), dtype=torch.uint8, device=dev)
    q_scales = torch.empty((q_rows, q_cols // 32), dtype=torch.uint8, device=dev)
    q_reps = 20
    with torch.cuda.stream(s):
        for _ in range(3):
            mm.musemoe_quantize_mxfp4(q_w, q_codes, q_scales, q_rows, q_cols, s)
        q0, q1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        q0.record(s)
        for _ in range(q_reps):
            mm.musemoe_quantize_mxfp4(q_w, q_codes, q_scales, q_rows, q_cols, s)
        q1.record(s)
    torch.cuda.synchronize()
    q_us = q0.elapsed_time(q1) * 1e3 / q_reps
    n_el = q_rows * q_cols
    q_bytes = 2 * n_el + n_el // 2 + n_el // 32
    quant_mxfp4 = {"us_per_launch": q_us, "algorithmic_bytes": q_bytes,
                   "achieved_gbs": q_bytes / (q_us / 1e6) / 1e9,
                   "frac": q_bytes / (q_us / 1e6) / 1e9 / hbm_peak,
                   "note": f"w13 of 32 experts [{q_rows}, {q_cols}] bf16, {q_reps} launches"}
    del q_w, q_codes, q_scales

    # end to end through the public API with host buffers
    e2e_steps = max(20, min(2000, args.steps // 10))
    xh, sh = sets[0]["x_host"], sets[0]["stream_host"]
    oh = torch.empty((cfg.rows, cfg.hidden), dtype=torch.int16).pin_memory()
    for i in range(5):
        st_ = sets[i % WEIGHT_SETS]
        mm.musemoe_forward_host(handle, st_["w"], st_["x_host"], st_["stream_host"], oh,
                                cfg.rows, s)
    barrier()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        st_ = sets[i % WEIGHT_SETS]
        mm.musemoe_forward_host(handle, st_["w"], st_["x_host"], st_["stream_host"], oh,
                                cfg.rows, s)
    t_e2e = max_over_ranks(time.perf_counter() - t0, world, dev)
    del xh, sh
    e2e_value = whole_job_rate(world, cfg.rows, e2e_steps, t_e2e)
    h2d = cfg.rows * cfg.hidden * (2 + 4)
    d2h = cfg.rows * cfg.hidden * (4 + 2)

    health = mm.musemoe_poll_health(handle)
    mm.musemoe_destroy(handle)
    # the other forms and the verify workload: single-GPU lines, measured
    # once (the scaling runs skip them)
    bf16_experts = w4a4 = None
    buckets = None
    if world == 1:
        bf16_experts = bench_bf16_experts(dev, hbm_peak)
        w4a4 = bench_w4a4(dev)
        buckets = {"verify": bench_bucket(dev, "verify", mm.MUSEMOE_NVFP4, hbm_peak, 16, 15.0),
                   "large": bench_bucket(dev, "large", mm.MUSEMOE_FP8_W8A8, hbm_peak, 16, 15.0),
                   "stack": bench_stack(dev, hbm_peak)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r = run_oracle(steps=4, budget_s=20.0, threads=1)
        tot = sum(r["times"])
        ncores = os.cpu_count() or 1
        rm = run_oracle(steps=6, budget_s=10.0, threads=ncores)
        tm = sum(rm["times"])
        cpu = {"value": r["rows"] * len(r["times"]) / tot, "unit": "rows/s", "cores": 1,
               "kind": "oracle",
               "sample": f"{len(r['times'])} full decode steps of {r['rows']} rows "
                         f"({tot:.1f} s, plain C float64, one thread)",
               "openmp_all_cores": {"value": rm["rows"] * len(rm["times"]) / tm,
                                    "unit": "rows/s", "cores": ncores,
                                    "sample": f"{len(rm['times'])} steps, the OpenMP build of "
                                              f"the same C source on {ncores} threads"}}

    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e2m1xf16->f32 (MXFP4 experts), bf16 dense, fp32 router",
        "data": "synthetic (seeded generator, random-init weights of the workload's shapes)",
        "config": {"workload": "decode bucket: b=8 rows, H=5120, P=2048, I=1024, E=128, "
                               "top-8, sigmoid, multiplier 0.5, MXFP4 experts",
                   "rows_per_gpu": cfg.rows, "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: {WEIGHT_SETS} rotating weight sets of "
                         f"{set_bytes / 1e6:.0f} MB",
                   "cuda_graph": (f"{WEIGHT_SETS} forwards per graph" if not args.eager
                                  else False)},
        "step_spread": (dict(_stats(rep_us), note=f"per step: 200 replays of the "
                             f"{WEIGHT_SETS}-forward graph, each timed alone")
                        if rep_us else None),
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm_peak,
                     "peak_source": peak_src, "unit": "GB/s", "frac": achieved / hbm_peak,
                     "traffic": traffic,
                     "algorithmic_bytes_per_launch": kernel_bytes[dom]},
        "block": {"algorithmic_bytes_per_step": step_bytes,
                  "achieved_gbs": step_bytes / (ms_step / 1e3) / 1e9,
                  "frac": step_bytes / (ms_step / 1e3) / 1e9 / hbm_peak,
                  "expert_phase_gbs": expert_bytes / (expert_ms / 1e3) / 1e9,
                  "expert_phase_frac": expert_bytes / (expert_ms / 1e3) / 1e9 / hbm_peak,
                  "active_experts": sum(m["active_experts"] for m in model) / len(model),
                  "kernel_us": {k_: v * 1e3 for k_, v in kernel_ms.items()},
                  "kernel_share": share},
        "e2e": {"value": e2e_value, "unit": "rows/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": kernels * args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "health": "ok" if health == mm.MUSEMOE_OK else "fp16 range",
        "buckets": buckets,
        "next": {"attention_boundary": attn_boundary, "quantize_mxfp4": quant_mxfp4,
                 "bf16_experts": bf16_experts, "w4a4": w4a4},
    }
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


# ------------------------------------------------------------ reference arm

def bench_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    warm = max(3, args.warmup) if args.warmup < 3 else args.warmup
    # bound the whole run to a few minutes: one oracle step is a full 8-row
    # decode step (about five seconds on one core)
    w_run = run_oracle(steps=min(warm, 3), budget_s=60.0, threads=1)
    per = sum(w_run["times"]) / len(w_run["times"])
    k = max(1, min(args.steps, int(120.0 / max(per, 1e-3))))
    r = run_oracle(steps=k, budget_s=150.0, threads=1)
    tot = sum(r["times"])
    value = r["rows"] * len(r["times"]) / tot
    capped = (f"capped from {args.steps} to fit a few minutes; "
              if len(r["times"]) < args.steps else "")
    sample = (f"{len(r['times'])} full decode steps of {r['rows']} rows ({capped}"
              f"plain C float64, one thread)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s",
        "n_gpus": world, "steps": len(r["times"]), "warmup": warm,
        "ms_per_step": tot / len(r["times"]) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded generator, random-init weights of the workload's shapes)",
        "config": {"workload": "decode bucket: b=8 rows, H=5120, P=2048, I=1024, E=128, "
                               "top-8, sigmoid, multiplier 0.5, MXFP4 experts",
                   "rows_per_gpu": 8, "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    args = _args()
    if args.impl == "reference":
        bench_reference(args)
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()
