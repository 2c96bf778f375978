"""Benchmark of the fused MoE layer forward on GB300.

One step = one forward of the Mixtral-8x7B-shaped MoE layer (K=4096,
N=14336, E=8, top_k=2, bf16 weights and activations) at each batch size of
the sweep M in {1, 8, 64, 512, 4096, 8192}: route -> permute -> grouped
GEMM1+silu_and_mul -> grouped GEMM2 -> finalize, all in the CUDA library.
``value`` = tokens of all ranks / (max over ranks of the timed seconds).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config mixtral|qwen3|deepseek|tiny]
  python bench.py --impl reference ...   # the CPU oracle on a bounded sample

Multi-GPU: replicas only (each rank runs the same workload on its own GPU, no
collective on the data path; a barrier and a max-reduce of the timing only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE-layer tokens/s at M=1..8192 tokens; % of HBM / tensor-core roofline"
UNIT = "tokens/s"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d["bf16_tflops_sustained"],
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


# ------------------------------------------------------------------ distributed plumbing

def dist_init(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world, device="cuda"):
    """The slowest rank's time (replicas: the job ends when the last one does)."""
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(v, world, device="cuda"):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def aggregate(units_per_rank, seconds_per_rank):
    """Whole-job throughput: all ranks' units over the slowest rank's time."""
    return sum(units_per_rank) / max(seconds_per_rank)


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev=0):
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"moe_bench_clocks_{os.getpid()}_{dev}.csv")
        sel = []
        try:
            u = str(torch.cuda.get_device_properties(dev).uuid)
            sel = ["-i", u if u.startswith("GPU-") else "GPU-" + u]
        except Exception:
            pass
        self.cmd = ["nvidia-smi", *sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                    "-lms", "100"]

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(self.cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = [l.strip().split(",") for l in open(self.path) if l.count(",") >= 8]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for n, v in zip(names[1:], r[5:9]):
                if "Active" in v and "Not" not in v:
                    reasons.add(n)
        pw = [float(r[3]) for r in rows if r[3].strip().replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(pw) if pw else None}


# ------------------------------------------------------------------ workload

def make_workload(cfg_name, device, only_m=None, experts=0, mxfp8_act=False, mxfp4_path="a16"):
    import dataclasses
    import mixture_experts_layer_15_gb300 as moe
    cfg = synth.CONFIGS[cfg_name]
    if experts:
        kw = dict(E=experts)
        if cfg.n_group > 1:
            kw.update(n_group=min(cfg.n_group, experts // 2), topk_group=min(cfg.topk_group, experts // 2))
        cfg = dataclasses.replace(cfg, **kw)
    li = synth.make_layer(cfg, device)
    # MXFP4 weights with bf16 activations (W4A16) run on the block-scaled
    # tensor cores (each activation as two E4M3 terms, MOE_WEIGHTS_MXFP4_A16);
    # mxfp4_path="decode" takes the decode-to-bf16 kernel instead
    fmt = moe.MOE_WEIGHTS_BF16
    if cfg.weight_format == "mxfp4":
        fmt = moe.MOE_WEIGHTS_MXFP4 if mxfp4_path == "decode" else moe.MOE_WEIGHTS_MXFP4_A16
    if mxfp8_act and cfg.weight_format == "mxfp4":
        fmt = moe.MOE_WEIGHTS_MXFP4_A8
    layer = moe.MoELayer(K=cfg.K, N=cfg.N, E=cfg.E, top_k=cfg.top_k, w1=li.w1, w2=li.w2,
                         w1_scale=li.w1_scale, w2_scale=li.w2_scale, fmt=fmt,
                         route="softmax" if cfg.route == "softmax" else "sigmoid",
                         score_bias=li.score_bias, n_group=cfg.n_group, topk_group=cfg.topk_group,
                         routed_scaling_factor=cfg.routed_scaling_factor, ws1=li.ws1, ws2=li.ws2,
                         fused_finalize=True)
    sweep = cfg.m_sweep if not only_m else tuple(only_m)
    batches = {M: synth.make_tokens(cfg, M, device, li) for M in sweep}
    return cfg, li, layer, batches


def launches_per_forward(moe, cfg, layer, M, finalize="fused"):
    """Kernels one forward launches: the router and permute (mirroring the
    library's plan), the experts step as the library reports it
    (moe_experts_launches, from the plan the call uses), and the finalize pass
    or shared expert where they run."""
    w = max(1, min(32, 8192 // cfg.E))
    if M <= 64 and M * cfg.top_k <= 32 * w:
        n = 1                                                 # router + permute in one kernel
    elif M * cfg.top_k <= 32 * w:
        n = 2                                                 # router; single-chunk permute
    else:
        n = 5                                                 # router; count/scan/scatter/gather
    fused = finalize == "fused"
    n += moe.moe_experts_launches(layer.cw, M, cfg.top_k, fused)
    if not fused:
        n += 1                                                # finalize pass
    if cfg.shared_N:
        # the shared expert: the same grouped kernels with one group of M rows
        sw = moe.make_weights(moe.MOE_WEIGHTS_BF16, 1, cfg.K, layer.Ns, layer.ws1, layer.ws2)
        n += moe.moe_experts_launches(sw, M, 1, False)
    return n


def roofline_layer(cfg, M, touched, pk, sustained=False, routed_mult=1.0, routes=None):
    """Slower of touched-expert weight bytes at HBM bandwidth and FLOPs at
    the bf16 tensor peak (the routed experts' FLOPs at routed_mult x that
    peak: 2, the nominal fp8 : bf16 ratio, for MXFP8 activations); returns
    (seconds, bytes, flops, tensor seconds). The burst peak by default: the
    per-M calls are single calls timed in isolation. ``routes``: the routed
    rows (M * top_k unless some experts are not local)."""
    bpw = 2.0 if cfg.weight_format == "bf16" else (0.5 + 1.0 / 32.0)
    wbytes = touched * 3.0 * cfg.K * cfg.N * bpw
    R = M * cfg.top_k if routes is None else routes
    flops = 6.0 * cfg.K * cfg.N * R
    if cfg.shared_N:
        wbytes += 3.0 * cfg.K * cfg.shared_N * 2.0
        flops += 6.0 * cfg.K * cfg.shared_N * M
    tc = (pk["bf16_sus"] if sustained else pk["bf16"]) * 1e12
    fr = 6.0 * cfg.K * cfg.N * R
    t_tc = fr / (tc * routed_mult) + (flops - fr) / tc
    return max(wbytes / (pk["hbm"] * 1e9), t_tc), wbytes, flops, t_tc


def make_forward(moe, cfg, layer, batches, stream, finalize="fused"):
    """One layer forward at batch size M through the C ABI: route + permute,
    [shared expert], experts (GEMM1, GEMM2; ``ev`` brackets them) and the
    finalize: folded into GEMM2 (finalize="fused", moe_experts_fused_finalize)
    or as a pass of its own over gemm2_permuted (finalize="two-pass")."""
    def forward(M, ev=None):
        x, logits = batches[M]
        b = layer.buffers(M)
        rsf_r = layer.rsf if layer.method == moe.MOE_ROUTE_SIGMOID_GROUPED_TOPK else 1.0
        # the folded finalize on the block-scaled formats gathers the rows in
        # the experts (moe_experts_fused_finalize_x): the permute copies none
        gx = finalize == "fused" and layer.gathers_in_experts(M)
        side = finalize == "fused" and layer.overlap_shared
        if side:
            # the shared expert on a second stream writes out's start (f32)
            # beside the router, the permute and the routed experts' first launches
            if layer._side is None:
                layer._side = (torch.cuda.Stream(device=x.device), torch.cuda.Event(), torch.cuda.Event())
            sstream, ev_in, ev_sh = layer._side
            ev_in.record(torch.cuda.current_stream())
            sstream.wait_event(ev_in)
            moe.moe_shared_expert(layer.ws1, layer.ws2, cfg.K, layer.Ns, x, M, b.out, moe.MOE_DTYPE_F32,
                                  b.shared_ws, b.shared_ws.numel(), sstream)
            ev_sh.record(sstream)
        moe.moe_route_permute(logits, M, cfg.E, cfg.top_k, layer.method, layer.score_bias, layer.n_group,
                              layer.topk_group, rsf_r, b.topk_ids, b.topk_weights, layer.weights_dtype, None,
                              cfg.E, x, cfg.K, b.offsets, b.pmap, b.inverse, None if gx else b.x_perm, b.perm_ws,
                              b.perm_ws.numel())
        if layer.ws1 is not None and not side:
            moe.moe_shared_expert(layer.ws1, layer.ws2, cfg.K, layer.Ns, x, M, b.shared, layer.gemm2_dtype,
                                  b.shared_ws, b.shared_ws.numel())
        rsf = 1.0 if layer.method == moe.MOE_ROUTE_SIGMOID_GROUPED_TOPK else layer.rsf
        if ev is not None:
            ev[0].record(stream)
        if side:
            moe.moe_experts_fused_finalize_after(layer.cw, x if gx else b.x_perm, 1 if gx else 0, b.offsets, M,
                                                 cfg.top_k, b.topk_weights, layer.weights_dtype, b.inverse, rsf,
                                                 b.out, ev_sh, b.exp_ws, b.exp_ws.numel())
            if ev is not None:
                ev[1].record(stream)
            return
        if finalize == "fused" and gx:
            moe.moe_experts_fused_finalize_x(layer.cw, x, b.offsets, M, cfg.top_k, b.topk_weights,
                                             layer.weights_dtype, b.inverse, b.shared, layer.gemm2_dtype, rsf,
                                             b.out, b.exp_ws, b.exp_ws.numel())
            if ev is not None:
                ev[1].record(stream)
            return
        if finalize == "fused":
            moe.moe_experts_fused_finalize(layer.cw, b.x_perm, b.offsets, M, cfg.top_k, b.topk_weights,
                                           layer.weights_dtype, b.inverse, b.shared, layer.gemm2_dtype, rsf,
                                           b.out, b.exp_ws, b.exp_ws.numel())
            if ev is not None:
                ev[1].record(stream)
            return
        moe.moe_experts(layer.cw, b.x_perm, b.offsets, M, cfg.top_k, b.gemm2, layer.gemm2_dtype, 0, None,
                        layer.weights_dtype, None, None, layer.gemm2_dtype, 1.0, None, layer.out_dtype,
                        b.exp_ws, b.exp_ws.numel())
        if ev is not None:
            ev[1].record(stream)
        moe.moe_finalize(b.gemm2, layer.gemm2_dtype, b.gemm2.shape[0], b.topk_weights, layer.weights_dtype,
                         b.pmap, M, cfg.top_k, cfg.K, b.shared, layer.gemm2_dtype, rsf, b.out, layer.out_dtype)
    return forward


def warm_up(moe, layer, sweep, forward, warmup):
    for M in sweep:                                # allocate buffers outside any timing
        layer.buffers(M)
    for _ in range(warmup):
        for M in sweep:
            forward(M)
    torch.cuda.synchronize()
    st = moe.moe_get_error()
    if st != 0:
        raise RuntimeError(f"device error during warm-up: {moe.status_string(st)}")


def l2_scrub(buf):
    """Untimed L2 scrub between breakdown samples: a read of a 1 GB buffer.
    It evicts everything (dirty lines are written back here, outside the
    timed region) and leaves only clean lines behind, so the next sample
    starts from a cold L2 without paying for another buffer's write-back."""
    torch.sum(buf)


def graph_time(forward, M, stream, scrub, reps):
    """Median time of a CUDA-graph replay of one forward at M (launch costs
    removed), each replay after an L2 scrub; None if capture fails."""
    try:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            forward(M)
        stream.wait_stream(side)
        with torch.cuda.graph(g):
            forward(M)
        torch.cuda.synchronize()
    except Exception as e:                      # capture unsupported: report, do not fail the bench
        torch.cuda.synchronize()
        return None, f"{type(e).__name__}: {e}"[:200]
    ts = []
    for _ in range(reps):
        scrub()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) / 1e3)
    del g
    return statistics.median(ts), None


def timed_sweep(moe, cfg, layer, sweep, forward, steps, stream, pk, world=1, clocks=None, reps=20,
                graph_max_m=64):
    """K timed steps of the whole sweep, with CUDA events only around the timed
    region (events between the kernels of a forward would break their
    programmatic-dependent-launch chaining). Then a per-M breakdown: for each
    M, the median of ``reps`` single forwards (and single experts calls),
    each after an L2 scrub, each bracketed by events; for M <= graph_max_m
    also the median of CUDA-graph replays of the forward. Returns (seconds
    over all steps, per-M breakdown, GEMM FLOPs, GEMM seconds, clocks)."""
    touched = {M: int((layer.buffers(M).offsets.diff() > 0).sum().item()) for M in sweep}
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.start()
    t0.record(stream)
    for _ in range(steps):
        for M in sweep:
            forward(M)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop() if clocks is not None else None
    st = moe.moe_get_error()
    if st != 0:
        raise RuntimeError(f"device error in the timed region: {moe.status_string(st)}")
    secs = t0.elapsed_time(t1) / 1e3

    buf = torch.zeros(256 << 20, dtype=torch.float32, device=stream.device)     # 1 GB > L2
    scrub = lambda: l2_scrub(buf)
    per_m = []
    gemm_flops = gemm_secs = 0.0
    for M in sweep:
        tf, tg = [], []
        for r in range(reps):
            for which, acc in ((0, tf), (1, tg)):
                scrub()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                if which == 0:
                    e0.record(stream)
                    forward(M)
                    e1.record(stream)
                else:
                    forward(M, (e0, e1))
                torch.cuda.synchronize()
                acc.append(e0.elapsed_time(e1) / 1e3)
        tm, tgm = statistics.median(tf), statistics.median(tg)
        mult = 2.0 if layer.fmt == moe.MOE_WEIGHTS_MXFP4_A8 else 1.0
        troof, wbytes, flops, t_tc = roofline_layer(cfg, M, touched[M], pk, routed_mult=mult)
        gf = 6.0 * cfg.K * cfg.N * M * cfg.top_k
        gemm_flops += gf
        gemm_secs += tgm
        rec = {"M": M, "tokens_per_s": M / tm, "ms": tm * 1e3, "gemm_ms": tgm * 1e3,
               "touched_experts": touched[M], "roofline_ms": troof * 1e3,
               "roofline_frac": troof / tm,
               "bound": "hbm" if wbytes / (pk["hbm"] * 1e9) >= t_tc else "tensor",
               "gemm_tflops": gf / tgm / 1e12, "weight_bytes": wbytes, "gemm_flops": gf,
               "peak_kind": "burst (single calls timed in isolation)"}
        if M <= graph_max_m:
            tgr, err = graph_time(forward, M, stream, scrub, reps)
            if tgr is not None:
                rec["graph_ms"] = tgr * 1e3
                rec["graph_roofline_frac"] = troof / tgr
            else:
                rec["graph_error"] = err
        per_m.append(rec)
    st = moe.moe_get_error()
    if st != 0:
        raise RuntimeError(f"device error in the breakdown: {moe.status_string(st)}")
    del buf
    return secs, per_m, gemm_flops, gemm_secs, clk


def experts_step_desc(moe, cfg, layer, M):
    """What the dominant launch is for this layer at batch M (its launch count
    from the library's plan)."""
    if layer.fmt in (moe.MOE_WEIGHTS_MXFP4_A8, moe.MOE_WEIGHTS_MXFP4_A16):
        act = "bf16 activations as two E4M3 terms" if layer.fmt == moe.MOE_WEIGHTS_MXFP4_A16 else "MXFP8 activations"
        return (f"the experts step at the largest M on the block-scaled MMAs ({act}): the activation quantiser, "
                "GEMM1 + activation and GEMM2 with the folded finalize, three launches")
    n = moe.moe_experts_launches(layer.cw, M, cfg.top_k, True)
    return (f"the experts step at the largest M: grouped GEMM1 + silu_and_mul and GEMM2 with the "
            f"folded finalize, {'one fused launch' if n == 1 else f'{n} launches'}")


def roofline_objects(per_m, pk, traffic=None, mult=1.0, kernel=None):
    """The roofline report of one config's sweep, each regime against its own
    peak (burst figures: every per-M call is timed alone):
    - ``dominant``: the experts step at the largest M (the launch that takes
      the most time): its algorithmic FLOPs (6 K N per routed row) over its
      event-timed duration, against the tensor peak;
    - ``hbm``: the HBM-bound batch sizes together: touched-expert weight bytes
      over the whole forward's time, against the measured HBM bandwidth."""
    big = max(per_m, key=lambda r: r["M"])
    peak_t = pk["bf16"] * mult
    ach = big["gemm_flops"] / (big["gemm_ms"] * 1e-3) / 1e12
    dom = {"kernel": kernel or "the experts step (grouped GEMM1 + activation, GEMM2, folded finalize)",
           "M": big["M"], "bound": "tensor", "achieved": ach, "peak": peak_t, "unit": "TFLOP/s",
           "frac": ach / peak_t,
           "peak_kind": f"{pk['src']} bf16 burst" + (" x 2 (fp8)" if mult != 1.0 else ""),
           "traffic": traffic, "algorithmic": "6*K*N*routes FLOPs of the experts step at the largest M"}
    hb = [r for r in per_m if r["bound"] == "hbm"]
    out = {"dominant": dom}
    if hb:
        gbs = sum(r["weight_bytes"] for r in hb) / (sum(r["ms"] for r in hb) * 1e-3) / 1e9
        out["hbm"] = {"M": [r["M"] for r in hb], "bound": "hbm", "achieved": gbs, "peak": pk["hbm"],
                      "unit": "GB/s", "frac": gbs / pk["hbm"], "peak_kind": f"{pk['src']} HBM copy",
                      "algorithmic": "touched-expert weight bytes of each whole forward"}
    return out


def other_config(moe, name, args, pk, dev, stream, cpu=False):
    """The same measurement on another config (reported beside the headline),
    with the oracle baseline on the host cores when ``cpu``."""
    cfg, li, layer, batches = make_workload(name, dev, mxfp4_path=args.mxfp4_path)
    sweep = sorted(batches)
    forward = make_forward(moe, cfg, layer, batches, stream, args.finalize)
    warm_up(moe, layer, sweep, forward, 3)
    steps = max(5, args.steps // 5)
    secs, per_m, gf, gs, _ = timed_sweep(moe, cfg, layer, sweep, forward, steps, stream, pk)
    wf = cfg.weight_format + " weights"
    if cfg.weight_format == "mxfp4":
        wf += (", bf16 activations decoded" if args.mxfp4_path == "decode" else
               ", bf16 activations as two E4M3 terms on block-scaled MMAs (W4A16)")
    out = {"workload": f"{cfg.name}-shaped MoE layer (K={cfg.K}, N={cfg.N}, E={cfg.E}, top_k={cfg.top_k}, "
                       f"{wf}{', shared expert' if cfg.shared_N else ''})",
           "tokens_per_s": sum(sweep) * steps / secs, "steps": steps, "gemm_tflops": gf / gs / 1e12,
           "roofline": roofline_objects(per_m, pk),
           "sweep": [{k: (round(v, 4) if isinstance(v, float) else v) for k, v in r.items()} for r in per_m]}
    if cpu:
        out["cpu_baseline"] = cpu_baselines(cfg, li, batches)
    del layer, li, batches
    torch.cuda.empty_cache()
    return out


def masked_stress(moe, pk, dev, stream, M=4096):
    """The deferred-finalize / masked-expert stress workload: the
    Qwen3-shaped layer at M = 4096 with a seeded random half of the 128
    experts non-local (their routes are -1 in the permute map), run as route +
    permute, the experts with do_finalize = 0 (gemm2_permuted, f32), then a
    separate finalize with a shared-expert output added (a seeded [M, K]
    tensor standing in for the shared expert's output). Median of 20 forwards,
    each after an L2 scrub; roofline over the local experts' routes."""
    import mixture_experts_layer_15_gb300 as _m
    cfg = synth.CONFIGS["qwen3"]
    li = synth.make_layer(cfg, dev)
    em, E_l = synth.masked_expert_map(cfg.E, seed=cfg.seed)
    keep = torch.from_numpy(np.nonzero(em.numpy() >= 0)[0]).to(dev)
    layer = moe.MoELayer(K=cfg.K, N=cfg.N, E=cfg.E, top_k=cfg.top_k, w1=li.w1[keep].contiguous(),
                         w2=li.w2[keep].contiguous(), expert_map=em.to(dev), E_local=E_l)
    x, logits = synth.make_tokens(cfg, M, dev, li)
    del li
    g = torch.Generator(device=dev).manual_seed(77)
    shared = torch.randn(M, cfg.K, generator=g, device=dev)
    F = _m.MOE_DTYPE_F32

    def fwd():
        b = layer.forward(x, logits, do_finalize=False)
        moe.moe_finalize(b.gemm2, F, b.gemm2.shape[0], b.topk_weights, F, b.pmap, M, cfg.top_k, cfg.K, shared, F,
                         1.0, b.out, F)
    for _ in range(3):
        fwd()
    torch.cuda.synchronize()
    buf = torch.zeros(256 << 20, dtype=torch.float32, device=dev)
    t = _median_time(fwd, stream, lambda: l2_scrub(buf))
    st = moe.moe_get_error()
    if st != 0:
        raise RuntimeError(f"device error in the masked stress row: {moe.status_string(st)}")
    b = layer.buffers(M)
    touched = int((b.offsets.diff() > 0).sum().item())
    R = int(b.offsets[-1].item())
    troof, wbytes, flops, t_tc = roofline_layer(cfg, M, touched, pk, routes=R)
    del buf, layer, x, logits, shared
    torch.cuda.empty_cache()
    return {"workload": f"qwen3-shaped layer, M={M}, expert_map with {E_l} of {cfg.E} experts local, "
                        "do_finalize=0, then moe_finalize with a shared-output add (f32)",
            "ms": t * 1e3, "tokens_per_s": M / t, "local_routes": R, "touched_local_experts": touched,
            "roofline_ms": troof * 1e3, "frac": troof / t, "peak_kind": "burst",
            "bound": "hbm" if wbytes / (pk["hbm"] * 1e9) >= t_tc else "tensor"}


def _median_time(fn, stream, scrub, reps=20):
    """Median CUDA-event time of fn() on `stream`, each call after an L2 scrub."""
    ts = []
    for _ in range(reps):
        scrub()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) / 1e3)
    return statistics.median(ts)


def next_rows(moe, pk, dev, stream):
    """The rows built beyond the core path, each timed on its own at a full
    size and set against its roofline: the finalize folded into the next
    layer's residual add + RMSNorm (HBM-bound: k rows of gemm2_permuted, the
    residual read and written, y written, all f32)."""
    out = {}
    buf = torch.zeros(256 << 20, dtype=torch.float32, device=dev)
    scrub = lambda: l2_scrub(buf)
    F = moe.MOE_DTYPE_F32
    rows = []
    for name in ("mixtral", "qwen3"):
        cfg = synth.CONFIGS[name]
        M, k, K = 8192, cfg.top_k, cfg.K
        g = torch.Generator(device=dev).manual_seed(11)
        g2 = torch.randn(M * k, K, generator=g, device=dev)
        w = torch.rand(M, k, generator=g, device=dev)
        pmap = torch.randperm(M * k, generator=g, device=dev).to(torch.int32).reshape(M, k)
        res = torch.randn(M, K, generator=g, device=dev)
        gamma = torch.rand(K, generator=g, device=dev) + 0.5
        y = torch.empty(M, K, device=dev)
        call = lambda: moe.moe_finalize_add_rmsnorm(g2, F, M * k, w, F, pmap, M, k, K, None, F, 1.0, res, F, gamma,
                                                    F, 1e-6, y, F)
        call()
        torch.cuda.synchronize()
        t = _median_time(call, stream, scrub)
        nbytes = M * k * K * 4 + M * k * 8 + M * K * 12 + K * 4
        rows.append({"workload": f"{name}-shaped, M={M}, top_k={k}, K={K}, f32", "ms": t * 1e3,
                     "algorithmic_bytes": nbytes, "achieved_gbs": nbytes / t / 1e9,
                     "frac": nbytes / t / 1e9 / pk["hbm"], "bound": "hbm"})
        del g2, w, pmap, res, gamma, y
    out["finalize_add_rmsnorm"] = rows

    # gelu_and_mul + activation_clamp in GEMM1's epilogue: the experts step
    # (tensor-bound) on the Mixtral-shaped layer, beside the same step with SiLU
    cfg = synth.CONFIGS["mixtral"]
    M = 4096
    li = synth.make_layer(cfg, dev)
    x, logits = synth.make_tokens(cfg, M, dev, li)
    batches = {M: (x, logits)}
    act_rows = []
    for act, clamp in (("silu", None), ("gelu", 1.0)):
        layer = moe.MoELayer(K=cfg.K, N=cfg.N, E=cfg.E, top_k=cfg.top_k, w1=li.w1, w2=li.w2, activation=act,
                             activation_clamp=clamp)
        fwd = make_forward(moe, cfg, layer, batches, stream, "fused")
        for _ in range(3):
            fwd(M)
        torch.cuda.synchronize()
        ts = []
        for _ in range(20):
            scrub()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            fwd(M, (e0, e1))
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / 1e3)
        t = statistics.median(ts)
        flops = 6.0 * cfg.K * cfg.N * M * cfg.top_k
        act_rows.append({"workload": f"mixtral-shaped experts step, M={M}, {act}_and_mul"
                                     + (f", clamp {clamp}" if clamp else ""),
                         "ms": t * 1e3, "tflops": flops / t / 1e12, "frac": flops / t / 1e12 / pk["bf16"],
                         "bound": "tensor", "peak_kind": "bf16 burst"})
        del layer
    out["activation"] = act_rows

    # the BatchedExperts layout: [E, max_tokens, K] with every block full
    T = 512
    w = moe.make_weights(moe.MOE_WEIGHTS_BF16, cfg.E, cfg.K, cfg.N, li.w1, li.w2)
    xb = torch.randn(cfg.E, T, cfg.K, device=dev).to(torch.bfloat16)
    counts = torch.full((cfg.E,), T, dtype=torch.int32, device=dev)
    yb = torch.empty(cfg.E, T, cfg.K, device=dev)
    wsb = torch.zeros(max(moe.moe_experts_batched_workspace_size(w, T), 16), dtype=torch.uint8, device=dev)
    call = lambda: moe.moe_experts_batched(w, xb, counts, T, yb, moe.MOE_DTYPE_F32, wsb, wsb.numel())
    call()
    torch.cuda.synchronize()
    t = _median_time(call, stream, scrub)
    flops = 6.0 * cfg.K * cfg.N * cfg.E * T
    out["batched_experts"] = [{"workload": f"mixtral-shaped, E={cfg.E}, max_tokens={T}, all blocks full, f32 out",
                               "ms": t * 1e3, "tflops": flops / t / 1e12, "frac": flops / t / 1e12 / pk["bf16"],
                               "bound": "tensor", "peak_kind": "bf16 burst"}]
    del xb, counts, yb, wsb
    del li, x, logits, batches
    torch.cuda.empty_cache()
    out["mxfp4_paths"] = a8_rows(moe, pk, dev, stream, scrub,
                                 fmts=(moe.MOE_WEIGHTS_MXFP4, moe.MOE_WEIGHTS_MXFP4_A16, moe.MOE_WEIGHTS_MXFP4_A8))
    del buf
    torch.cuda.empty_cache()
    return out


def a8_rows(moe, pk, dev, stream, scrub, sweep=(1, 64, 1024, 8192), fmts=None):
    """The DeepSeek-shaped layer with its MXFP4 routed experts on MXFP8
    activations (block-scaled MMAs, MOE_WEIGHTS_MXFP4_A8) beside the same
    layer on bf16 activations: the whole forward (route + permute, shared
    expert, experts with the folded finalize) per M, median of 20 scrubbed
    runs, and the experts step alone. Roofline: touched weight bytes at HBM
    bandwidth vs FLOPs at the tensor peak of each path's MMAs (the routed
    experts at the fp8 peak = measured bf16 burst x 2, the nominal
    fp8 : bf16 ratio, on the A8 path; bf16 otherwise; the shared expert bf16;
    burst peaks, since every forward is timed alone)."""
    cfg = synth.CONFIGS["deepseek"]
    li = synth.make_layer(cfg, dev)
    batches = {M: synth.make_tokens(cfg, M, dev, li) for M in sweep}
    rows = []
    tags = {moe.MOE_WEIGHTS_MXFP4: "bf16 activations (decode to bf16, kind::f16)",
            moe.MOE_WEIGHTS_MXFP4_A16: "bf16 activations as two E4M3 terms (kind::mxf8f6f4 block-scaled)",
            moe.MOE_WEIGHTS_MXFP4_A8: "MXFP8 activations (kind::mxf8f6f4 block-scaled)"}
    for fmt in (fmts or (moe.MOE_WEIGHTS_MXFP4, moe.MOE_WEIGHTS_MXFP4_A8)):
        tag = tags[fmt]
        layer = moe.MoELayer(K=cfg.K, N=cfg.N, E=cfg.E, top_k=cfg.top_k, w1=li.w1, w2=li.w2,
                             w1_scale=li.w1_scale, w2_scale=li.w2_scale, fmt=fmt, route="sigmoid",
                             score_bias=li.score_bias, n_group=cfg.n_group, topk_group=cfg.topk_group,
                             routed_scaling_factor=cfg.routed_scaling_factor, ws1=li.ws1, ws2=li.ws2)
        fwd = make_forward(moe, cfg, layer, batches, stream, "fused")
        for M in sweep:
            for _ in range(3):
                fwd(M)
        torch.cuda.synchronize()
        for M in sweep:
            tf, tg = [], []
            for _ in range(20):
                for which, acc in ((0, tf), (1, tg)):
                    scrub()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    if which == 0:
                        e0.record(stream)
                        fwd(M)
                        e1.record(stream)
                    else:
                        fwd(M, (e0, e1))
                    torch.cuda.synchronize()
                    acc.append(e0.elapsed_time(e1) / 1e3)
            t, tgm = statistics.median(tf), statistics.median(tg)
            touched = int((layer.buffers(M).offsets.diff() > 0).sum().item())
            wbytes = touched * 3.0 * cfg.K * cfg.N * (0.5 + 1.0 / 32.0) + 3.0 * cfg.K * cfg.shared_N * 2.0
            fr = 6.0 * cfg.K * cfg.N * M * cfg.top_k
            fs = 6.0 * cfg.K * cfg.shared_N * M
            p_routed = pk["bf16"] * (2.0 if fmt == moe.MOE_WEIGHTS_MXFP4_A8 else 1.0) * 1e12
            t_tc = fr / p_routed + fs / (pk["bf16"] * 1e12)
            t_hbm = wbytes / (pk["hbm"] * 1e9)
            troof = max(t_tc, t_hbm)
            rows.append({"workload": f"deepseek-shaped layer, M={M}, {tag}", "M": M, "ms": t * 1e3,
                         "experts_ms": tgm * 1e3, "experts_tflops": fr / tgm / 1e12,
                         "tokens_per_s": M / t, "roofline_ms": troof * 1e3, "frac": troof / t,
                         "bound": "hbm" if t_hbm >= t_tc else "tensor"})
        st = moe.moe_get_error()
        if st != 0:
            raise RuntimeError(f"device error in the MXFP8 rows: {moe.status_string(st)}")
        del layer, fwd
        torch.cuda.empty_cache()
    del li, batches
    torch.cuda.empty_cache()
    return rows


def run_gpu(args):
    import mixture_experts_layer_15_gb300 as moe
    rank, world = dist_init(args.gpus)
    dev = torch.device("cuda", torch.cuda.current_device())
    pk = peaks()
    stream = torch.cuda.current_stream()
    cfg, li, layer, batches = make_workload(args.config, dev, args.m, args.experts, args.mxfp8_act, args.mxfp4_path)
    sweep = sorted(batches)
    forward = make_forward(moe, cfg, layer, batches, stream, args.finalize)
    warm_up(moe, layer, sweep, forward, args.warmup)
    clocks = ClockSampler(torch.cuda.current_device())
    secs, per_m, gemm_flops, gemm_secs, clk = timed_sweep(moe, cfg, layer, sweep, forward, args.steps, stream,
                                                          pk, world, clocks)
    secs_max = max_over_ranks(secs, world)
    tokens_step = sum(sweep)
    value = tokens_step * args.steps * world / secs_max
    traffic = tcase = talg = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    big_m = max(sweep)
    if os.path.exists(tpath) and not (args.experts or args.mxfp8_act) and args.finalize == "fused":
        try:
            t = json.load(open(tpath)).get(args.config) or {}
            if t.get("M") == big_m:            # counters of the launch the roofline describes
                traffic, tcase, talg = t.get("bytes_per_launch"), t.get("case"), t.get("algorithmic_bytes")
        except Exception:
            traffic = None
    objs = roofline_objects(per_m, pk, traffic=traffic, kernel=experts_step_desc(moe, cfg, layer, big_m))
    roof = dict(objs["dominant"])
    roof.update(traffic_case=tcase, traffic_algorithmic=talg)

    e2e = run_e2e(args, cfg, layer, batches, forward_fn=forward)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": secs_max / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{cfg.name}-shaped MoE layer (K={cfg.K}, N={cfg.N}, E={cfg.E}, "
                               f"top_k={cfg.top_k}, {cfg.weight_format} weights), one forward at each M",
                   "M_sweep": sweep, "tokens_per_step": tokens_step,
                   "storage": "f32 routing weights, gemm2_permuted and output; bf16 act",
                   "finalize": ("folded into the GEMM2 epilogue (f32 reductions into out; gemm2_permuted not "
                                "materialised)" if args.finalize == "fused" else
                                "separate pass over gemm2_permuted (deterministic order)"),
                   "l2": "timed steps: inputs larger than L2 (expert weights streamed every forward); per-M breakdown: a 1 GB read scrub before each sample (median of 20)",
                   "parallelism": f"replicas x{world}"},
        "roofline": roof, "roofline_hbm": objs.get("hbm"), "sweep": per_m, "e2e": e2e,
        "gpu_launches": args.steps * sum(launches_per_forward(moe, cfg, layer, M, args.finalize) for M in sweep),
        "clocks": clk,
    }
    if rank == 0:
        line["cpu_baseline"] = None if args.no_cpu_baseline else cpu_baselines(cfg, li, batches)
        if args.others and not args.m and not args.experts and not args.mxfp8_act:
            del layer, batches
            torch.cuda.empty_cache()
            line["other_configs"] = {name: other_config(moe, name, args, pk, dev, stream,
                                                        cpu=not args.no_cpu_baseline)
                                     for name in args.others.split(",") if name and name != args.config}
            line["masked_stress"] = masked_stress(moe, pk, dev, stream)
            line["next_rows"] = next_rows(moe, pk, dev, stream)
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(args, cfg, layer, batches, forward_fn):
    """Same metric through the public API with host buffers: every step copies
    each batch's x and router logits from pinned host memory to the device
    and reads each output back. Three streams pipeline the step: the H2D copy
    of a batch, its forward, and the D2H copy of its output; events keep each
    buffer from being reused before its previous user is done."""
    comp = torch.cuda.current_stream()
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    Ms = sorted(batches)
    host = {M: (x.cpu().pin_memory(), lg.cpu().pin_memory()) for M, (x, lg) in batches.items()}
    outs = {M: torch.empty(layer.buffers(M).out.shape, dtype=layer.buffers(M).out.dtype).pin_memory()
            for M in Ms}
    dev_in = {M: (torch.empty_like(x), torch.empty_like(lg)) for M, (x, lg) in batches.items()}
    ev = lambda: torch.cuda.Event()
    in_free = {M: ev() for M in Ms}      # forward of M has consumed its inputs
    in_ready = {M: ev() for M in Ms}     # inputs of M are on the device
    out_ready = {M: ev() for M in Ms}    # output of M computed
    out_free = {M: ev() for M in Ms}     # output of M copied back
    for M in Ms:
        in_free[M].record(comp)
        out_free[M].record(comp)
    orig = dict(batches)
    steps = max(3, args.steps // 4)
    h2d = sum(x.numel() * x.element_size() + lg.numel() * lg.element_size() for x, lg in host.values())
    d2h = sum(o.numel() * o.element_size() for o in outs.values())
    try:
        for M in Ms:
            batches[M] = dev_in[M]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for it in range(2 + steps):
            if it == 2:
                torch.cuda.synchronize()
                t0.record(comp)
                h2d_s.wait_event(t0)                    # no timed copy starts before t0
                d2h_s.wait_event(t0)
            for M in Ms:
                h2d_s.wait_event(in_free[M])
                with torch.cuda.stream(h2d_s):
                    dev_in[M][0].copy_(host[M][0], non_blocking=True)
                    dev_in[M][1].copy_(host[M][1], non_blocking=True)
                in_ready[M].record(h2d_s)
                comp.wait_event(in_ready[M])
                comp.wait_event(out_free[M])
                forward_fn(M)
                in_free[M].record(comp)
                out_ready[M].record(comp)
                d2h_s.wait_event(out_ready[M])
                with torch.cuda.stream(d2h_s):
                    outs[M].copy_(layer.buffers(M).out, non_blocking=True)
                out_free[M].record(d2h_s)
            if it == 1 + steps:
                for M in Ms:
                    comp.wait_event(out_free[M])         # the step ends when its outputs are on the host
        t1.record(comp)
        torch.cuda.synchronize()
    finally:
        batches.update(orig)
    secs = t0.elapsed_time(t1) / 1e3
    return {"value": sum(Ms) * steps / secs, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps,
            "pipelining": "H2D, compute and D2H on three streams; every step copies all its inputs and outputs"}


# ------------------------------------------------------------------ CPU oracle

class _F64Experts:
    """Per-expert float64 weights for the oracle. bf16 weights are converted
    once, outside the timing; MXFP4 bytes are dequantised by the oracle on
    every access (its own step from the packed bytes), unless ``cache``."""

    def __init__(self, w, scale=None, cache=None):
        import oracle as O
        self.cache = {}
        self.keep = scale is None if cache is None else cache
        self.w, self.scale, self.O = w, scale, O

    def __getitem__(self, e):
        if e in self.cache:
            return self.cache[e]
        if self.scale is None:
            v = self.w[e].to(torch.float64).cpu().numpy()
        else:
            v = self.O.dequant_mxfp4(self.w[e].cpu().numpy(), self.scale[e].cpu().numpy())
        if self.keep:
            self.cache[e] = v
        return v

    @property
    def shape(self):
        s = tuple(self.w.shape)
        return s if self.scale is None else s[:-1] + (s[-1] * 2,)


def _oracle_forward(O, cfg, li, w1, w2, x, logits):
    return O.moe_forward(x, logits, w1, w2, cfg.top_k,
                         route="softmax" if cfg.route == "softmax" else "sigmoid",
                         score_bias=None if li.score_bias is None else li.score_bias.cpu().numpy(),
                         n_group=cfg.n_group, topk_group=cfg.topk_group,
                         routed_scaling_factor=cfg.routed_scaling_factor,
                         ws1=None if li.ws1 is None else li.ws1.double().cpu().numpy(),
                         ws2=None if li.ws2 is None else li.ws2.double().cpu().numpy())["out"]


def _oracle_setup(cfg, li, batches):
    import oracle as O
    w1, w2 = _F64Experts(li.w1, li.w1_scale), _F64Experts(li.w2, li.w2_scale)
    Mbig = max(batches)
    x, logits = batches[Mbig]
    xs = x.to(torch.float64).cpu().numpy()
    ls = logits.cpu().numpy()
    if li.w1_scale is None:
        ids, _ = (O.route_softmax_topk(ls[:256], cfg.top_k) if cfg.route == "softmax" else
                  O.route_sigmoid_grouped(ls[:256], li.score_bias.cpu().numpy(), cfg.top_k, cfg.n_group,
                                          cfg.topk_group, cfg.routed_scaling_factor))
        for e in sorted(set(ids.reshape(-1).tolist())):   # convert the bf16 weights the sample uses, untimed
            w1[e], w2[e]
    return O, w1, w2, xs, ls


def _blas_threads(n=None):
    """Get (n None) or set the thread count of the OpenBLAS that numpy loaded,
    through the setter it exports; None if no such library or symbol."""
    import ctypes
    libs = set()
    for line in open("/proc/self/maps"):
        f = line.split()[-1]
        if f.startswith("/") and "openblas" in os.path.basename(f).lower():
            libs.add(f)
    for path in sorted(libs):
        lib = ctypes.CDLL(path)
        for pre in ("scipy_openblas", "openblas"):
            for suf in ("64_", "_64", ""):
                get, put = f"{pre}_get_num_threads{suf}", f"{pre}_set_num_threads{suf}"
                if hasattr(lib, get) and hasattr(lib, put):
                    if n is None:
                        return int(getattr(lib, get)())
                    getattr(lib, put)(ctypes.c_int(n))
                    return n
    return None


def _time_oracle(cfg, li, batches, budget_s):
    """The oracle, as it stands, on the first S tokens of the largest batch
    through the whole layer; S grows until a run takes about budget_s / 4."""
    O, w1, w2, xs, ls = _oracle_setup(cfg, li, batches)
    n = min(xs.shape[0], 4096)
    S, secs = min(n, 1 if li.w1_scale is not None else 4), 0.0
    while True:
        t = time.perf_counter()
        _oracle_forward(O, cfg, li, w1, w2, xs[:S], ls[:S])
        secs = time.perf_counter() - t
        if secs * 4 > budget_s or S >= n:
            break
        S = min(n, S * (2 if li.w1_scale is not None else 4))
    return S, secs


def cpu_baselines(cfg, li, batches, budget_s=12.0):
    """The oracle (numpy float64) timed on the host cores on a bounded sample
    of this config's largest batch: with every core numpy's BLAS uses, and on
    one core (BLAS set to one thread, the calling thread pinned to one CPU).
    MXFP4 experts are dequantised by the oracle inside the timing."""
    what = ("including the oracle's dequantisation of every touched MXFP4 expert"
            if li.w1_scale is not None else "bf16 weights converted to float64 beforehand")
    S, secs = _time_oracle(cfg, li, batches, budget_s)
    n_all = _blas_threads() or os.cpu_count()
    out = {"value": S / secs, "unit": UNIT, "cores": n_all, "kind": "oracle",
           "sample": f"first {S} tokens of the M={max(batches)} {cfg.name} batch through the whole layer "
                     f"(numpy float64, {what}), {secs:.2f} s"}
    prev_aff = os.sched_getaffinity(0)
    prev_thr = _blas_threads()
    try:
        set_ok = _blas_threads(1) == 1
        os.sched_setaffinity(0, {min(prev_aff)})
        S1, secs1 = _time_oracle(cfg, li, batches, budget_s)
    finally:
        os.sched_setaffinity(0, prev_aff)
        if prev_thr:
            _blas_threads(prev_thr)
    out["one_core"] = {"value": S1 / secs1, "unit": UNIT, "cores": 1 if set_ok else None, "kind": "oracle",
                       "sample": f"first {S1} tokens, {secs1:.2f} s, one CPU "
                                 + ("(BLAS set to one thread)" if set_ok else
                                    "(BLAS thread count could not be set: cores not known)")}
    return out


def run_reference(args):
    """--impl reference: the CPU oracle timed on the host cores, each step a
    bounded sample of the same workload; rank 0 only."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    cfg = synth.CONFIGS[args.config]
    li = synth.make_layer(cfg, dev)
    batches = {M: synth.make_tokens(cfg, M, dev, li) for M in cfg.m_sweep}
    O, w1, w2, xs, ls = _oracle_setup(cfg, li, batches)
    # size the per-step sample so the whole run stays within ~2 minutes
    t = time.perf_counter()
    _oracle_forward(O, cfg, li, w1, w2, xs[:2], ls[:2])
    per_tok = max((time.perf_counter() - t) / 2, 1e-4)
    S = int(max(1, min(64, 120.0 / (args.steps + args.warmup) / per_tok)))
    for _ in range(args.warmup):
        _oracle_forward(O, cfg, li, w1, w2, xs[:S], ls[:S])
    t = time.perf_counter()
    for s in range(args.steps):
        o = (s * S) % max(1, xs.shape[0] - S)
        _oracle_forward(O, cfg, li, w1, w2, xs[o:o + S], ls[o:o + S])
    secs = time.perf_counter() - t
    value = S * args.steps / secs
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": f"{cfg.name}-shaped MoE layer (K={cfg.K}, N={cfg.N}, E={cfg.E}, "
                                   f"top_k={cfg.top_k}, {cfg.weight_format} weights), one forward at each M",
                       "M_sweep": list(cfg.m_sweep)},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"{S} tokens of the M={max(cfg.m_sweep)} batch per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="mixtral", choices=sorted(synth.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--m", type=int, nargs="*", default=None,
                    help="run only these batch sizes of the sweep (profiling)")
    ap.add_argument("--finalize", default="fused", choices=["fused", "two-pass"],
                    help="finalize folded into GEMM2 (f32 reductions, order not fixed) or a separate pass")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing (profiling)")
    ap.add_argument("--others", default="qwen3,deepseek",
                    help="other configs measured after the headline one and reported beside it ('' = none)")
    ap.add_argument("--experts", type=int, default=0,
                    help="profiling only: keep the first N experts of the config (not the benchmark workload)")
    ap.add_argument("--mxfp4-path", default="a16", choices=["a16", "decode"],
                    help="MXFP4 weights with bf16 activations: on the block-scaled MMAs (two E4M3 terms per "
                         "activation) or decoded to bf16 in shared memory")
    ap.add_argument("--mxfp8-act", action="store_true",
                    help="profiling only: MXFP4 configs run their experts on MXFP8 activations "
                         "(MOE_WEIGHTS_MXFP4_A8; not the benchmark workload)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
