"""Multi-rank logic on CPU ranks (gloo, world size 2).

* Expert parallelism: rank r owns experts [r E/g, (r+1) E/g). Routing, the
  pooler and the pre-expert norm are replicated; each rank runs its own
  experts on the routes that select them, applies the post-expert norm and
  the router weight per route (both are per route, so they stay local), and
  the ranks all-reduce (sum) the partial moe_out [b, P]. Unpooler and FFN
  boundary are replicated. The result must equal the single-process block.
* The bench's whole-job timing: the max over ranks of the timed region and
  the weak-scaling rate built from it.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORLD = 2


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank: int, world: int, port: int):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _ep_rank(rank: int, world: int, port: int, cfg_name: str, result):
    _init(rank, world, port)
    try:
        import oracle as O
        import synth
        cfg = synth.CONFIGS[cfg_name]
        w = synth.layer_tensors(cfg)
        x, st = synth.activations(cfg)
        rp = synth.routing_params(cfg)
        E = cfg.experts
        lo, hi = rank * E // world, (rank + 1) * E // world
        # replicated front: router, routing, pooler + pre-expert norm
        logits = O.router_logits(x, w["w_router"])
        r = O.route(logits, w["expert_bias"], rp["top_k"], rp["route_scale"], rp["multiplier"],
                    rp["score"], rp["division_eps"])
        h = O.pre_expert(x, w["w_pool"], w["w_pre_norm"], cfg.norm_eps, True)
        # local experts only: a route whose expert lives elsewhere contributes 0
        local = (r.ids >= lo) & (r.ids < hi)
        y = np.zeros((cfg.rows, cfg.top_k, cfg.pooled))
        for e in range(lo, hi):
            tok, slot = np.nonzero(r.ids == e)
            if tok.size:
                one = np.full((tok.size, 1), e, dtype=np.int32)
                y[tok, slot] = O.expert_outputs(h[tok], one, cfg.quant, w, cfg.inter)[:, 0]
        n = O.rms_norm(y, O.bf16_to_f64(w["w_post_norm"]), cfg.norm_eps)
        part = (n * r.weights[..., None] * local[..., None]).sum(axis=1)
        t = torch.from_numpy(part)
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        moe_out = O.round_bf16(t.numpy())
        u = O.unpool(moe_out, w["w_unpool"])
        s_new, out = O.boundary(u, st, w["w_ffn_norm"], float(w["gate"][0]), w["w_next_norm"],
                                cfg.norm_eps)
        result[rank] = dict(moe_out=moe_out, stream=s_new, out=out,
                            local_routes=int(local.sum()))
    finally:
        dist.destroy_process_group()


def _timing_rank(rank: int, world: int, port: int, result):
    _init(rank, world, port)
    try:
        import bench
        ms = 10.0 + 5.0 * rank                      # rank 1 is the slow one
        m = bench.max_over_ranks(ms, world)
        result[rank] = (m, bench.whole_job_rate(world, 8, 100, m / 1e3))
    finally:
        dist.destroy_process_group()


def _spawn(fn, *args):
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        result = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=fn, args=(r, WORLD, port, *args, result))
                 for r in range(WORLD)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=300)
        codes = [p.exitcode for p in procs]
        for p in procs:
            if p.is_alive():
                p.kill()
        assert codes == [0] * WORLD, codes
        return dict(result)


@pytest.mark.parametrize("cfg_name", ["tiny", "edge_tiny", "w4a4_tiny", "w4a4_nv_tiny"])
def test_expert_parallel_matches_single_process(cfg_name):
    sys.path.insert(0, ROOT)
    import oracle as O
    import synth
    cfg = synth.CONFIGS[cfg_name]
    res = _spawn(_ep_rank, cfg_name)
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    ref = O.block(x, st, w, quant=cfg.quant, norm_eps=cfg.norm_eps,
                  **synth.routing_params(cfg))
    # every route ran on exactly one rank
    assert res[0]["local_routes"] + res[1]["local_routes"] == cfg.rows * cfg.top_k
    assert res[0]["local_routes"] > 0 and res[1]["local_routes"] > 0
    for r in range(WORLD):
        # the partial sums add in another order: equal to fp64 rounding, and
        # identical after the bf16 rounding of moe_out
        np.testing.assert_array_equal(res[r]["moe_out"], ref["moe_out"])
        np.testing.assert_array_equal(res[r]["stream"], ref["stream"])
        np.testing.assert_array_equal(res[r]["out"], ref["out"])


def test_bench_timing_takes_slowest_rank():
    res = _spawn(_timing_rank)
    for r in range(WORLD):
        m, rate = res[r]
        assert m == 15.0
        assert rate == pytest.approx(WORLD * 8 * 100 / 0.015)


def _ep_rank_library(rank: int, world: int, port: int, cfg_name: str, result):
    """A rank of the expert-parallel block through the library on cuda:0: its
    experts' partial moe_out (musemoe_forward_ep_partial), the all-reduce over
    gloo (host tensors), then musemoe_forward_ep_combine. The ranks' kernels
    never wait on one another: they meet only in the host all-reduce."""
    _init(rank, world, port)
    try:
        import dataclasses

        import moe_decode_layer_router_gb300 as mm
        import synth
        from tests import _harness as H
        torch.cuda.set_device(0)
        mm.library()
        cfg = synth.CONFIGS[cfg_name]
        w = synth.layer_tensors(cfg)
        x, st = synth.activations(cfg)
        E = cfg.experts
        lo, hi = rank * E // world, (rank + 1) * E // world
        keys = ("w13", "w13_scale", "w13_gscale", "w2", "w2_scale", "w2_gscale")
        t = {k: H.to_dev(v) for k, v in w.items() if k not in keys}
        for k in keys:
            if k in w:
                t[k] = H.to_dev(np.ascontiguousarray(w[k][lo:hi]))
        mm.musemoe_pack_experts(H.dims_of(dataclasses.replace(cfg, experts=hi - lo)),
                                H.QUANT[cfg.quant], t["w13"], t.get("w13_scale"), t["w13"],
                                t.get("w13_scale"), t["w2"], t.get("w2_scale"), t["w2"],
                                t.get("w2_scale"))
        W = mm.make_weights(t)
        run = H.Run(cfg)
        try:
            part = torch.empty((cfg.rows, cfg.pooled), dtype=torch.float32, device="cuda")
            mm.musemoe_forward_ep_partial(run.handle, W, H.to_dev(x), part, cfg.rows, lo, hi - lo)
            torch.cuda.synchronize()
            host = part.cpu()
            dist.all_reduce(host, op=dist.ReduceOp.SUM)
            sd = H.to_dev(st)
            out = torch.empty((cfg.rows, cfg.hidden), dtype=torch.int16, device="cuda")
            mm.musemoe_forward_ep_combine(run.handle, W, host.cuda(), sd, out, cfg.rows)
            torch.cuda.synchronize()
            ok = mm.musemoe_poll_health(run.handle) == mm.MUSEMOE_OK
        finally:
            run.close()
        result[rank] = dict(stream=sd.cpu().numpy().astype(np.float64),
                            out=out.cpu().numpy().view(np.uint16).copy(), ok=ok)
    finally:
        dist.destroy_process_group()


@pytest.mark.gpu
@pytest.mark.parametrize("cfg_name", ["tiny", "decode"])
def test_expert_parallel_library_on_two_ranks(cfg_name):
    sys.path.insert(0, ROOT)
    import oracle as O
    import synth
    from tests import _harness as H
    cfg = synth.CONFIGS[cfg_name]
    res = _spawn(_ep_rank_library, cfg_name)
    w = synth.layer_tensors(cfg)
    x, st = synth.activations(cfg)
    ref = O.block(x, st, w, quant=cfg.quant, norm_eps=cfg.norm_eps,
                  **synth.routing_params(cfg))
    # both ranks hold the same all-reduced block output, within the block's bounds
    np.testing.assert_array_equal(res[0]["out"], res[1]["out"])
    np.testing.assert_array_equal(res[0]["stream"], res[1]["stream"])
    assert res[0]["ok"] and res[1]["ok"]
    assert H.rel_err(res[0]["stream"], ref["stream"]) <= H.OUT_TOL
    assert H.rel_err(O.bf16_to_f64(res[0]["out"]), ref["out"]) <= H.OUT_TOL
