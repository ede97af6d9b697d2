"""Benchmark of the MoE layer forward on GB300 (one JSON line on rank 0).

A step is one moe_forward over one batch of T synthetic tokens (router logits, top-k,
counts/offsets/permutation, dispatch, the grouped SwiGLU expert GEMMs, combine), with the
inputs and weights resident in HBM. L2 is flushed (a 512 MB write) before every timed step
and each step is timed with CUDA events on the launching stream. Per-stage times come from
a second loop over the staged entry points, timed the same way.

The headline is the Mixtral-shaped layer (T=4096, H=4096, 8 experts top-2, F=14336). The
default run then measures the other four layer shapes the same way (tiny fp32,
DeepSeek-V3-shaped bf16, imbalanced routing, FP8 dispatch), and the FP8 shape with MXFP8
block scales, and reports them under "configs", each with its throughput, its grouped-GEMM
and dispatch/combine rooflines and its own CPU-oracle baseline (--headline-only skips them).

  python bench.py [--gpus N --steps K --warmup W] [--workload NAME] [--impl reference]

Multi-GPU: independent token-sharded replicas (no collective in the data path; the path has
no exchange step on one node), launched with torch.distributed.run; value = tokens of all
ranks / max-over-ranks time. --impl reference times the CPU oracle on a bounded token
sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

DEFAULT_WORKLOAD = "mixtral_bf16"
L2_FLUSH_BYTES = 512 << 20


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def rank_env():
    """(world, rank, local_rank) from the torch.distributed.run environment."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def shard_seed(rank: int) -> int:
    """Each replica draws its own token shard; the weights use seed 0 on every rank."""
    return rank


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The largest value over all ranks (the job's time is its slowest replica's)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_rank: int, steps: int, max_ms: float) -> float:
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank * steps / (max_ms / 1e3)


def describe(w):
    return (f"{w['name']} (T={w['T']}, H={w['H']}, E={w['E']}, k={w['k']}, F={w['F']}"
            + (f", shared F={w['F_shared']}" if w["n_shared"] else "")
            + (f", groups {w['topk_groups']}/{w['n_groups']}" if w["n_groups"] > 1 else "")
            + (", e4m3 transfer (1x128 / 128x128 fp32 scales)" if w["xfer_dtype"] == synth.E4M3 else "")
            + (", MXFP8 transfer (e4m3, 1x32 UE8M0 scales)" if w["xfer_dtype"] == synth.MXE4M3 else "") + ")")


def quant_kind(w):
    """0 unquantised, 1 FP8 with fp32 block scales, 2 MXFP8."""
    return {synth.E4M3: 1, synth.MXE4M3: 2}.get(w["xfer_dtype"], 0)


# DRAM bytes (read + write) per forward of the two grouped-GEMM launches, from one-pass ncu
# captures (dram__bytes_read.sum + dram__bytes_write.sum) of the current GEMM kernels on the
# full-size workloads. A workload without an entry has no capture of the current kernels and
# reports null.
_SRC = "one-pass ncu capture (dram__bytes_read.sum + dram__bytes_write.sum) of GEMM1 + GEMM2, full-size workload"
GEMM_TRAFFIC = {
    "mixtral_bf16": (2.08e9 + 0.23054e9 + 1.50e9 + 0.06014e9, _SRC),
    "dsv3_bf16": (17.67e9 + 0.29932e9 + 7.89e9 + 1.02e9, _SRC),
    "imbalanced_bf16": (1.45e9 + 0.19702e9 + 0.57717e9 + 0.51493e9, _SRC),
    "dsv3_fp8": (13.39e9 + 0.66015e9 + 4.96e9 + 4.20e9, _SRC),
    "dsv3_mxfp8": (13.618e9 + 0.62394e9 + 5.149e9 + 4.2014e9, _SRC),
    "tiny_fp32": (2.379e6 + 1.584e6, _SRC),
}


def gemm_traffic(w):
    t = GEMM_TRAFFIC.get(w["name"])
    return {"traffic": t[0], "traffic_source": t[1]} if t else {"traffic": None}


def algorithmic(w):
    """Algorithmic bytes / flops per forward (each tensor read or written once)."""
    T, H, E, k, F = w["T"], w["H"], w["E"], w["k"], w["F"]
    R = T * k
    a = 4 if w["act_dtype"] == synth.F32 else 2
    qk = quant_kind(w)
    x8 = qk != 0
    xs = 1 if x8 else a
    shared = T if w["n_shared"] else 0
    d = {}
    d["gemm_flops"] = synth.gemm_flops(w)
    d["router_flops"] = 2.0 * T * H * E
    # x read once, the k (+1 shared) rows written, tok_row read, and the scales written:
    # fp32 per 1x128 block, or one UE8M0 byte per 1x32 block (plus the expert ids read)
    d["dispatch_bytes"] = T * H * a + (R + (shared if x8 else 0)) * H * xs + R * 4 \
        + ((R + shared) * (H // 128) * 4 if qk == 1 else 0) + ((R + shared) * (H // 32) + R * 4 if qk == 2 else 0)
    d["combine_bytes"] = (R + shared) * H * a + T * H * a + R * 8
    d["weight_bytes"] = (E * 3 * F * H + (3 * w["F_shared"] * H if w["n_shared"] else 0)) * xs
    return d


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


class GpuContext:
    """The rank's device, peaks, stream and L2-flush buffer, shared by every workload."""

    def __init__(self):
        import torch
        self.world, self.rank, local = rank_env()
        self.dist = None
        if self.world > 1:
            import torch.distributed as dist
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
            self.dist = dist
        else:
            torch.cuda.set_device(0)
        self.dev = torch.device("cuda", torch.cuda.current_device())
        self.peaks, self.peak_kind = load_peaks()
        self.flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=self.dev)
        self.stream = torch.cuda.current_stream()

    def barrier(self):
        import torch
        torch.cuda.synchronize()
        if self.dist is not None:
            self.dist.barrier()
        torch.cuda.synchronize()


def build_layer(ctx, w):
    """This rank's token shard (seed = rank) and the replicated weights (seed 0) of workload
    w, drawn on the device; e4m3 / MX weights quantised once, outside any timing."""
    import torch
    import token_routing_expert_router_gb300 as moe
    dev = ctx.dev
    dt = torch.bfloat16 if w["act_dtype"] == synth.BF16 else torch.float32
    T, H, E, k, F = w["T"], w["H"], w["E"], w["k"], w["F"]
    s = w["w_std"]

    def gen(shape, tid, std, seed=0, dtype=dt):
        t = torch.empty(shape, dtype=dtype, device=dev)
        return synth.device_normal(t, seed, tid, std)

    x = gen((T, H), synth.X, 1.0, seed=shard_seed(ctx.rank))
    wts = {"w_router": gen((E, H), synth.W_ROUTER, s), "w_gate": gen((E, F, H), synth.W_GATE, s),
           "w_up": gen((E, F, H), synth.W_UP, s), "w_down": gen((E, H, F), synth.W_DOWN, s),
           "router_bias": torch.from_numpy(synth.zipf_bias(0, E)).to(dev) if w["zipf"] else None}
    if w["n_shared"]:
        Fs = w["F_shared"]
        wts["ws_gate"] = gen((Fs, H), synth.WS_GATE, s)
        wts["ws_up"] = gen((Fs, H), synth.WS_UP, s)
        wts["ws_down"] = gen((H, Fs), synth.WS_DOWN, s)
    qk = quant_kind(w)
    if qk:
        pairs = [("w_gate", "s_gate"), ("w_up", "s_up"), ("w_down", "s_down")]
        if w["n_shared"]:
            pairs += [("ws_gate", "ss_gate"), ("ws_up", "ss_up"), ("ws_down", "ss_down")]
        for wn, sn in pairs:
            src = wts[wn].reshape(-1, wts[wn].shape[-1])
            q = torch.empty(src.shape, dtype=torch.uint8, device=dev)
            if qk == 2:
                sc = torch.empty((src.shape[0] // 128) * (src.shape[1] // 128) * 512, dtype=torch.uint8, device=dev)
                moe.moe_quantize_mx(src, q, sc)
            else:
                sc = torch.empty((src.shape[0] // 128, src.shape[1] // 128), dtype=torch.float32, device=dev)
                moe.moe_quantize_e4m3(src, 128, 128, q, sc)
            wts[wn] = q.reshape(wts[wn].shape)
            wts[sn] = sc
            del src
    cfg = moe.MoEConfig.make(**{kk: w[kk] for kk in (
        "T", "H", "E", "k", "F", "n_shared", "F_shared", "score_fn", "renorm", "n_groups",
        "topk_groups", "group_score", "routed_scale", "act_dtype", "xfer_dtype")})
    ws = torch.zeros(moe.moe_forward_workspace_size(cfg) // 4 + 64, dtype=torch.int32, device=dev)
    moe.moe_workspace_init(ws)
    y = torch.empty((T, H), dtype=dt, device=dev)
    return {"w": w, "cfg": cfg, "x": x, "wts": wts, "ws": ws, "y": y, "dt": dt, "gen": gen}


def time_forward(ctx, L, steps, warmup, use_graph=True):
    """W warm-up forwards, then K forwards (CUDA-graph replays of moe_forward), each after an
    L2-flushing write and bracketed by CUDA events on the launching stream, with nvidia-smi
    sampling the clocks meanwhile; then the same steps with L2 left warm (context)."""
    import torch
    import token_routing_expert_router_gb300 as moe
    cfg, x, wts, y, ws = L["cfg"], L["x"], L["wts"], L["y"], L["ws"]
    stream = ctx.stream
    for _ in range(warmup):
        moe.moe_forward(cfg, x, wts, y, ws)
    st = moe.moe_read_status(ws)
    assert st == moe.MOE_OK, moe.moe_status_string(st)
    graph = None
    if use_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            moe.moe_forward(cfg, x, wts, y, ws)
        graph.replay()
    step = graph.replay if graph is not None else (lambda: moe.moe_forward(cfg, x, wts, y, ws))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    ctx.barrier()
    with ClockSampler(torch.cuda.current_device()) as clocks:
        t_wall = time.perf_counter()
        for i in range(steps):
            ctx.flush.fill_(float(i))  # evict the previous step's lines from L2
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        ctx.barrier()
        t_wall = time.perf_counter() - t_wall
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(step_ms), ctx.dist, ctx.dev)
    assert moe.moe_read_status(ws) == moe.MOE_OK
    n_warm = max(3, min(steps, 20))
    ev_w = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_warm)]
    step()
    for i in range(n_warm):
        ev_w[i][0].record(stream)
        step()
        ev_w[i][1].record(stream)
    torch.cuda.synchronize()
    warm_ms = statistics.median(a.elapsed_time(bb) for a, bb in ev_w)
    del graph
    return {"total_ms": total_ms, "ms_per_step": total_ms / steps, "wall_s": t_wall, "clocks": clocks.summary(),
            "warm_ms": warm_ms, "used_graph": use_graph}


def stage_buffers(ctx, L):
    import torch
    import token_routing_expert_router_gb300 as moe
    w, cfg, dev, dt = L["w"], L["cfg"], ctx.dev, L["dt"]
    T, H, E, k, F = w["T"], w["H"], w["E"], w["k"], w["F"]
    R = T * k
    rows = R + (T if w["n_shared"] else 0)
    qk = quant_kind(w)
    xdt = torch.uint8 if qk else dt

    def act_scales(K):
        if qk == 2:
            return torch.empty(moe.moe_mx_scale_bytes(cfg, K), dtype=torch.uint8, device=dev)
        return torch.empty((K // 128, rows), dtype=torch.float32, device=dev) if qk == 1 else None

    return {"logits": torch.empty((T, E), dtype=torch.float32, device=dev),
            "idx": torch.empty((T, k), dtype=torch.int32, device=dev),
            "w": torch.empty((T, k), dtype=torch.float32, device=dev),
            "counts": torch.empty(E, dtype=torch.int32, device=dev),
            "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
            "row_token": torch.empty(R, dtype=torch.int32, device=dev),
            "tok_row": torch.empty((T, k), dtype=torch.int32, device=dev),
            "xd": torch.empty((rows, H), dtype=xdt, device=dev),
            "xd_scale": act_scales(H),
            "h": torch.empty((rows, F), dtype=xdt, device=dev),
            "h_scale": act_scales(F),
            "yd": torch.empty((rows, H), dtype=dt, device=dev)}


def time_stages(ctx, L, b, reps, gather=True):
    """Each staged entry point (the same kernels moe_forward launches) as one call after an
    L2 flush, median of ``reps``; dispatch and combine again with L2 warm (context)."""
    import torch
    import token_routing_expert_router_gb300 as moe
    w, cfg, x, wts, ws, y = L["w"], L["cfg"], L["x"], L["wts"], L["ws"], L["y"]
    qk = quant_kind(w)
    stream = ctx.stream
    stages = {
        "router_logits": lambda: moe.moe_router_logits(cfg, x, wts["w_router"], wts["router_bias"], b["logits"], ws),
        "route": lambda: moe.moe_route(cfg, b["logits"], b["idx"], b["w"], b["counts"], b["offsets"],
                                       b["row_token"], b["tok_row"], ws),
        "dispatch": (lambda: moe.moe_dispatch_mx(cfg, x, b["idx"], b["tok_row"], b["offsets"], b["xd"],
                                                 b["xd_scale"])) if qk == 2 else
                    (lambda: moe.moe_dispatch(cfg, x, b["tok_row"], b["xd"], b["xd_scale"])),
        "grouped_mlp": lambda: moe.moe_grouped_mlp(cfg, b["xd"], b["xd_scale"], x, b["offsets"], wts, b["h"],
                                                   b["h_scale"], b["yd"], ws),
        "combine": lambda: moe.moe_combine(cfg, b["yd"], b["tok_row"], b["w"], y),
    }
    if gather and w["act_dtype"] == synth.BF16 and not qk:  # the fused-permutation alternative
        # rows gathered by token in GEMM1, routing weights applied in GEMM2's epilogue
        stages["grouped_mlp_gather"] = lambda: moe.moe_grouped_mlp_gather(cfg, x, b["row_token"], b["offsets"],
                                                                          wts, b["h"], b["yd"], ws,
                                                                          tok_row=b["tok_row"], topk_w=b["w"])
    for _ in range(2):
        for f in stages.values():
            f()
    times = {n: [] for n in stages}
    for _ in range(reps):
        for n, f in stages.items():
            ctx.flush.fill_(1.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            f()
            e1.record(stream)
            times[n].append((e0, e1))
    torch.cuda.synchronize()
    assert moe.moe_read_status(ws) == moe.MOE_OK
    stage_ms = {n: statistics.median(a.elapsed_time(bb) for a, bb in v) for n, v in times.items()}
    warm = {}
    for n in ("dispatch", "combine"):  # again without the flush: the call's own inputs warm in L2
        f = stages[n]
        f()
        pairs = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            f()
            e1.record(stream)
            pairs.append((e0, e1))
        torch.cuda.synchronize()
        warm[n] = statistics.median(a.elapsed_time(bb) for a, bb in pairs)
    return stage_ms, warm


def back_to_back(ctx, make_buffers, call, nbytes):
    """Per-launch time of K launches replayed back to back from one CUDA graph, each on its
    own copy of the inputs and outputs (together well beyond L2, flushed first), so the
    per-launch time leaves out the launch and completion overhead that a single timed
    ~15 us launch carries, without any launch finding the previous one's data in L2."""
    import torch
    K = max(3, min(8, -(-600_000_000 // max(1, nbytes))))
    bufs = [make_buffers() for _ in range(K)]
    for bb in bufs:  # warm
        call(bb)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()  # the K launches replay from one graph: no host pacing
    with torch.cuda.graph(g):
        for bb in bufs:
            call(bb)
    torch.cuda.synchronize()
    ms = []
    for _ in range(3):
        ctx.flush.fill_(3.0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(ctx.stream)
        g.replay()
        e1.record(ctx.stream)
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1) / K)
    del g, bufs
    torch.cuda.empty_cache()
    return statistics.median(ms), K


def time_dispatch_combine(ctx, L, b, alg):
    import torch
    import token_routing_expert_router_gb300 as moe
    cfg, x, y = L["cfg"], L["x"], L["y"]
    qk = quant_kind(L["w"])

    def dispatch_bufs():
        return {"x": x.clone(), "xd": torch.empty_like(b["xd"]),
                "xs": torch.empty_like(b["xd_scale"]) if b["xd_scale"] is not None else None}

    def dispatch_call(bb):
        if qk == 2:
            moe.moe_dispatch_mx(cfg, bb["x"], b["idx"], b["tok_row"], b["offsets"], bb["xd"], bb["xs"])
        else:
            moe.moe_dispatch(cfg, bb["x"], b["tok_row"], bb["xd"], bb["xs"])

    def combine_bufs():
        return {"yd": b["yd"].clone(), "y": torch.empty_like(y)}

    disp, k_disp = back_to_back(ctx, dispatch_bufs, dispatch_call, alg["dispatch_bytes"])
    comb, k_comb = back_to_back(ctx, combine_bufs, lambda bb: moe.moe_combine(cfg, bb["yd"], b["tok_row"], b["w"],
                                                                              bb["y"]), alg["combine_bytes"])
    return disp, k_disp, comb, k_comb


def tensor_peak(ctx, w, kind="bf16_tflops"):
    """The measured bf16 peak of the given kind (burst for calls timed alone), times the
    part's nominal fp8:bf16 dense ratio of 2 for the e4m3 GEMMs."""
    p = ctx.peaks.get(kind, ctx.peaks["bf16_tflops"])
    return p * (2.0 if quant_kind(w) else 1.0)


def fp32_alu_peak(ctx):
    """fp32 FMA peak derived from unit counts and clocks: SMs x 128 FMA lanes per clock x 2
    flops x the maximum SM clock (the fp32 grouped GEMM runs on the SIMT pipes)."""
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    mhz = ctx.peaks.get("sm_max_mhz", 2070.0)
    return sms * 128 * 2 * mhz * 1e6 / 1e12, f"derived: {sms} SMs x 128 fp32 FMA/clk x 2 flops x {mhz:.0f} MHz"


def gemm_roofline(ctx, w, gemm_ms, alg):
    achieved = alg["gemm_flops"] / (gemm_ms / 1e3) / 1e12
    if w["act_dtype"] == synth.F32:
        peak, kind = fp32_alu_peak(ctx)
        return {"kernel": "SIMT fp32 grouped GEMM (gate/up + SwiGLU, down): 2 launches per forward",
                "bound": "alu", "achieved": round(achieved, 2), "peak": round(peak, 1), "peak_kind": kind,
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                "timing": "CUDA events around moe_grouped_mlp on the launching stream, median of the stage loop",
                **gemm_traffic(w)}
    peak = tensor_peak(ctx, w)
    sus = tensor_peak(ctx, w, "bf16_tflops_sustained")
    out = {"kernel": "tc grouped GEMM (gate/up + SwiGLU, down): 2 launches per forward",
           "bound": "tensor", "achieved": round(achieved, 1), "peak": round(peak, 1),
           "peak_kind": f"{ctx.peak_kind} bf16 burst" + (" x2 (nominal fp8:bf16 dense ratio)" if quant_kind(w) else "")
                        + ": the GEMM pair is timed as single calls after an L2 flush",
           "unit": "TFLOP/s", "frac": round(achieved / peak, 3),
           "frac_of_sustained": round(achieved / sus, 3),
           "timing": "CUDA events around moe_grouped_mlp on the launching stream, median of the stage loop",
           **gemm_traffic(w)}
    # the other roof: the recorded DRAM traffic over the same time, against the measured copy rate
    # (the DeepSeek-V3 shapes stream their weights once, so this one binds as much as the tensor's)
    if out.get("traffic"):
        gbs = out["traffic"] / (gemm_ms / 1e3) / 1e9
        out["dram_gbs"] = round(gbs, 1)
        out["dram_frac"] = round(gbs / ctx.peaks["hbm_gbs"], 3)
        out["weight_bound_ms"] = round(alg["weight_bytes"] / (ctx.peaks["hbm_gbs"] * 1e9) * 1e3, 3)
    return out


def hbm_roofline(ctx, alg, disp_ms, comb_ms):
    d = alg["dispatch_bytes"] / (disp_ms / 1e3) / 1e9
    c = alg["combine_bytes"] / (comb_ms / 1e3) / 1e9
    return {"dispatch_gbs": round(d, 1), "combine_gbs": round(c, 1),
            "dispatch_frac": round(d / ctx.peaks["hbm_gbs"], 3), "combine_frac": round(c / ctx.peaks["hbm_gbs"], 3),
            "peak_gbs": ctx.peaks["hbm_gbs"], "peak_kind": ctx.peak_kind + " copy (read + write)"}


def config_of(w, world):
    """The workload's config object, the same for both arms."""
    return {"workload": describe(w), "tokens_per_gpu": w["T"], "parallelism": f"replicas x{world} (token-sharded)",
            "weights_bytes": algorithmic(w)["weight_bytes"]}


def dtype_name(w):
    return {1: "e4m3+bf16", 2: "mxfp8(e4m3,ue8m0)+bf16"}.get(quant_kind(w), "bf16" if w["act_dtype"] == synth.BF16 else "f32")


# Oracle tokens per workload for the CPU baseline: about 2-20 s of fp64 work each on a
# 16-core host (the DeepSeek-V3 shapes touch most of their experts' weights even for a few
# tokens, and drawing those weights on the host is not timed but takes time).
CPU_TOKENS = {"tiny_fp32": 256, "mixtral_bf16": 64, "dsv3_bf16": 8, "imbalanced_bf16": 64, "dsv3_fp8": 8,
              "dsv3_mxfp8": 8}
OTHER_CONFIGS = ["tiny_fp32", "dsv3_bf16", "imbalanced_bf16", "dsv3_fp8", "dsv3_mxfp8"]


def measure_config(ctx, args, w):
    """One workload's forward, stages, GEMM roofline and dispatch/combine rooflines (the
    entries of the "configs" object)."""
    import torch
    L = build_layer(ctx, w)
    steps = max(3, min(args.steps, 20))
    fw = time_forward(ctx, L, steps, args.warmup, use_graph=not args.no_graph)
    b = stage_buffers(ctx, L)
    stage_ms, warm = time_stages(ctx, L, b, reps=max(3, min(args.steps, 10)), gather=False)
    alg = algorithmic(w)
    disp, _, comb, _ = time_dispatch_combine(ctx, L, b, alg)
    counts = b["counts"].cpu().numpy()
    T = w["T"]
    out = {"workload": describe(w), "dtype": dtype_name(w),
           "value": round(job_tokens_per_s(ctx.world, T, steps, fw["total_ms"]), 1), "unit": "tokens/s",
           "ms_per_step": round(fw["ms_per_step"], 4), "steps": steps,
           "stages_ms": {n: round(v, 4) for n, v in stage_ms.items()},
           "grouped_gemm": gemm_roofline(ctx, w, stage_ms["grouped_mlp"], alg),
           "dispatch_combine": dict(hbm_roofline(ctx, alg, disp, comb), dispatch_ms=round(disp, 4),
                                    combine_ms=round(comb, 4)),
           "expert_rows": {"min": int(counts.min()), "max": int(counts.max()), "empty": int((counts == 0).sum())},
           "clocks": fw["clocks"]}
    if w["T"] <= 512:
        out["note"] = "launch-latency-bound layer: the roofline fractions carry little meaning"
    del L, b
    torch.cuda.empty_cache()
    if ctx.rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w, min(CPU_TOKENS.get(w["name"], args.cpu_tokens), T))
    return out


def run_gpu(args, w):
    import torch
    import token_routing_expert_router_gb300 as moe

    ctx = GpuContext()
    moe.build()
    L = build_layer(ctx, w)
    cfg, x, wts, ws, y, dt, gen = L["cfg"], L["x"], L["wts"], L["ws"], L["y"], L["dt"], L["gen"]
    dev, stream, flush, dist = ctx.dev, ctx.stream, ctx.flush, ctx.dist
    T, H, E, k, F = w["T"], w["H"], w["E"], w["k"], w["F"]
    world, rank = ctx.world, ctx.rank

    # ---- whole-layer steps (moe_forward issues no host sync, so one step is a CUDA graph)
    fw = time_forward(ctx, L, args.steps, args.warmup, use_graph=not args.no_graph)
    ms_per_step = fw["ms_per_step"]
    value = job_tokens_per_s(world, T, args.steps, fw["total_ms"])

    # ---- per-stage times through the staged entry points (same kernels)
    qk = quant_kind(w)
    fp8 = qk != 0
    b = stage_buffers(ctx, L)
    stage_ms, warm_stage = time_stages(ctx, L, b, reps=max(3, min(args.steps, 10)))
    alg = algorithmic(w)
    b2b_disp, k_disp, b2b_comb, k_comb = time_dispatch_combine(ctx, L, b, alg)

    # ---- end to end: pinned host x in, host y out, through moe_forward_host. Two streams,
    # each with its own workspace, device staging and pinned buffers, take the steps in turn,
    # so the copies of one step run under the kernels of the other; every step still makes
    # its own host->device copy of x and device->host copy of y inside the timed region.
    e2e_steps = max(4, min(args.steps, 20))
    # pinned buffers on the GPU's own host node: the process runs on the CPUs local to the
    # GPU while it allocates and uses them (best effort; restored afterwards)
    saved_affinity, local_cpus = set_gpu_local_affinity(dev)
    lanes = []
    for _ in range(2):
        wsl = torch.zeros(moe.moe_forward_workspace_size(cfg) // 4 + 64, dtype=torch.int32, device=dev)
        moe.moe_workspace_init(wsl)
        xh = torch.empty((T, H), dtype=dt, pin_memory=True)
        xh.copy_(x)
        lanes.append({"ws": wsl, "xh": xh, "yh": torch.empty((T, H), dtype=dt, pin_memory=True),
                      "xdev": torch.empty_like(x), "ydev": torch.empty_like(y), "s": torch.cuda.Stream(device=dev)})
    for ln in lanes:  # warm both lanes
        moe.moe_forward_host(cfg, ln["xh"], wts, ln["yh"], ln["xdev"], ln["ydev"], ln["ws"], stream=ln["s"])
    torch.cuda.synchronize()
    ctx.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for ln in lanes:
        ln["s"].wait_event(e0)
    for i in range(e2e_steps):
        ln = lanes[i % 2]
        moe.moe_forward_host(cfg, ln["xh"], wts, ln["yh"], ln["xdev"], ln["ydev"], ln["ws"], stream=ln["s"])
    for ln in lanes:
        stream.wait_stream(ln["s"])
    e1.record(stream)
    ctx.barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dist, dev)
    for ln in lanes:
        assert moe.moe_read_status(ln["ws"]) == moe.MOE_OK
    if saved_affinity is not None:
        os.sched_setaffinity(0, saved_affinity)

    # ---- backward (training step) of the same layer: bf16 layers
    bwd = None
    if not args.no_backward and w["act_dtype"] == synth.BF16 and not fp8:
        bwd = time_backward(args, w, cfg, x, wts, ws, b, flush, stream, gen, dev, dt)
    counts = b["counts"].cpu().numpy()
    h2d_bytes, d2h_bytes = int(x.numel() * x.element_size()), int(y.numel() * y.element_size())
    del L, b, x, y, wts, ws, lanes
    torch.cuda.empty_cache()

    # ---- the other layer shapes, each measured the same way (forward only)
    others = {}
    if not args.headline_only and not (args.tokens or args.experts):
        for name in OTHER_CONFIGS:
            if name != w["name"]:
                others[name] = measure_config(ctx, args, synth.WORKLOADS[name])

    if rank != 0:
        dist.destroy_process_group()
        return None
    roof = gemm_roofline(ctx, w, stage_ms["grouped_mlp"], alg)
    hbm = hbm_roofline(ctx, alg, b2b_disp, b2b_comb)
    line = {
        "metric": "MoE-layer fwd tokens/s",
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype_name(w),
        "data": "synthetic (seeded N(0,1) tokens, N(0,0.02^2) weights; no dataset or trained weights)",
        "config": config_of(w, world),
        "timing": {"l2": f"flushed before every timed step ({L2_FLUSH_BYTES >> 20} MB write)",
                   "launch": "CUDA graph replay of moe_forward" if fw["used_graph"] else "moe_forward calls"},
        "stages_ms": {n: round(v, 4) for n, v in stage_ms.items()},
        "warm_l2": {"note": "context only: L2 not flushed between calls, so inputs and weights may be served "
                            "from L2; the flushed numbers are the results",
                    "ms_per_step": round(fw["warm_ms"], 4), "tokens_per_s": round(T * world / (fw["warm_ms"] / 1e3), 1),
                    "dispatch_ms": round(warm_stage["dispatch"], 4), "combine_ms": round(warm_stage["combine"], 4),
                    "dispatch_gbs": round(alg["dispatch_bytes"] / (warm_stage["dispatch"] / 1e3) / 1e9, 1),
                    "combine_gbs": round(alg["combine_bytes"] / (warm_stage["combine"] / 1e3) / 1e9, 1)},
        "dispatch_gbs": hbm["dispatch_gbs"],
        "combine_gbs": hbm["combine_gbs"],
        "dispatch_combine_timing": {
            "method": "per launch, from K launches replayed back to back from one CUDA graph, each "
                      "on its own copy of its buffers (L2 flushed first, K copies well beyond L2)",
            "dispatch_ms": round(b2b_disp, 4), "dispatch_K": k_disp,
            "combine_ms": round(b2b_comb, 4), "combine_K": k_comb,
            "dispatch_gbs_single_launch": round(alg["dispatch_bytes"] / (stage_ms["dispatch"] / 1e3) / 1e9, 1),
            "combine_gbs_single_launch": round(alg["combine_bytes"] / (stage_ms["combine"] / 1e3) / 1e9, 1)},
        "grouped_gemm_tflops": roof["achieved"],
        "grouped_gemm_frac_of_peak": roof["frac"],
        "roofline": roof,
        "hbm_roofline": hbm,
        "expert_rows": {"min": int(counts.min()), "max": int(counts.max()), "empty": int((counts == 0).sum())},
        "e2e": {"value": round(job_tokens_per_s(world, T, 1, e2e_ms), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d_bytes,
                "d2h_bytes_per_step": d2h_bytes,
                "call": "moe_forward_host (pinned host x in, host y out), steps alternating on two streams",
                "host_cpus": local_cpus or "not restricted",
                "l2": "not flushed (each step's x arrives by its own host-to-device copy)"},
        "gpu_launches": args.steps * launches_per_forward(w),
        **({"backward": bwd} if bwd is not None else {}),
        "clocks": fw["clocks"],
        "wall_s_timed_region": round(fw["wall_s"], 3),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_tokens)
    if others:
        line["configs"] = others
    if dist is not None:
        dist.destroy_process_group()
    return line


def time_backward(args, w, cfg, x, wts, ws, b, flush, stream, gen, dev, dt):
    """The training step's backward: moe_backward_kept after moe_forward_train (the gate/up
    pre-activations kept, the router's backward and the auxiliary loss's gradient included).
    Beside it: the training forward, moe_backward (recomputing the gate/up GEMM) with and
    without the router, and the staged calls (combine backward, grouped MLP backward, router
    backward, the fused input gradient and the plain dispatch backward). L2 flushed before
    each call."""
    import torch
    import token_routing_expert_router_gb300 as moe
    T, H, E, k, F = w["T"], w["H"], w["E"], w["k"], w["F"]
    rows = T * k + (T if w["n_shared"] else 0)
    bws = torch.zeros(moe.moe_backward_workspace_size(cfg) // 4 + 64, dtype=torch.int32, device=dev)
    moe.moe_workspace_init(bws)
    dy = gen((T, H), synth.DY, 1.0)
    dx = torch.empty((T, H), dtype=dt, device=dev)
    dtw = torch.empty((T, k), dtype=torch.float32, device=dev)
    grads = {"dw_gate": torch.empty((E, F, H), dtype=torch.float32, device=dev),
             "dw_up": torch.empty((E, F, H), dtype=torch.float32, device=dev),
             "dw_down": torch.empty((E, H, F), dtype=torch.float32, device=dev)}
    if w["n_shared"]:
        Fs = w["F_shared"]
        grads.update(dws_gate=torch.empty((Fs, H), dtype=torch.float32, device=dev),
                     dws_up=torch.empty((Fs, H), dtype=torch.float32, device=dev),
                     dws_down=torch.empty((H, Fs), dtype=torch.float32, device=dev))
    rgrads = dict(grads, dw_router=torch.empty((E, H), dtype=torch.float32, device=dev),
                  dlogits=torch.empty((T, E), dtype=torch.float32, device=dev), aux_loss_coeff=0.01)
    if wts.get("router_bias") is not None:
        rgrads["d_router_bias"] = torch.empty((E,), dtype=torch.float32, device=dev)
    rws = torch.zeros(moe.moe_router_backward_workspace_size(cfg) // 4 + 64, dtype=torch.int32, device=dev)
    moe.moe_workspace_init(rws)
    dyd = torch.empty((rows, H), dtype=dt, device=dev)
    dxd = torch.empty((rows, H), dtype=dt, device=dev)
    gu = torch.empty((rows, 2 * F), dtype=dt, device=dev)
    yt = torch.empty((T, H), dtype=dt, device=dev)
    aux = torch.empty((1,), dtype=torch.float32, device=dev)
    moe.moe_forward_train(cfg, x, wts, yt, ws, gu, aux_alpha=0.01, aux_loss=aux)
    stages = {
        "backward": lambda: moe.moe_backward_kept(cfg, x, wts, dy, ws, gu, dx, dtw, rgrads, bws),
        "forward_train": lambda: moe.moe_forward_train(cfg, x, wts, yt, ws, gu, aux_alpha=0.01, aux_loss=aux),
        "forward_same_timing": lambda: moe.moe_forward(cfg, x, wts, yt, ws),
        "backward_recompute": lambda: moe.moe_backward(cfg, x, wts, dy, ws, dx, dtw, rgrads, bws),
        "backward_without_router": lambda: moe.moe_backward(cfg, x, wts, dy, ws, dx, dtw, grads, bws),
        "combine_backward": lambda: moe.moe_combine_backward(cfg, dy, b["yd"], b["tok_row"], b["w"], dyd, dtw),
        "grouped_mlp_backward": lambda: moe.moe_grouped_mlp_backward(cfg, b["xd"], x, b["offsets"], wts, dyd, dxd,
                                                                     grads, bws),
        "router_backward": lambda: moe.moe_router_backward(cfg, b["logits"], b["idx"], dtw, x, rgrads["dlogits"],
                                                           rgrads["dw_router"], rws,
                                                           d_router_bias=rgrads.get("d_router_bias"),
                                                           counts=b["counts"], aux_alpha=0.01),
        "dispatch_router_backward": lambda: moe.moe_dispatch_router_backward(cfg, dxd, b["tok_row"], rgrads["dlogits"],
                                                                             wts["w_router"], dx, rws),
        "dispatch_backward": lambda: moe.moe_dispatch_backward(cfg, dxd, b["tok_row"], dx),
    }
    for f in stages.values():
        f()
    moe.moe_forward_train(cfg, x, wts, yt, ws, gu, aux_alpha=0.01, aux_loss=aux)  # g and u match ws again

    # the whole training step (training forward + training backward) as one CUDA graph
    def train_step():
        moe.moe_forward_train(cfg, x, wts, yt, ws, gu, aux_alpha=0.01, aux_loss=aux)
        moe.moe_backward_kept(cfg, x, wts, dy, ws, gu, dx, dtw, rgrads, bws)

    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        train_step()
    torch.cuda.current_stream().wait_stream(side)
    tgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(tgraph):
        train_step()
    tgraph.replay()
    stages["training_step_graph"] = tgraph.replay
    reps = max(3, min(args.steps, 5))
    times = {n: [] for n in stages}
    for _ in range(reps):
        for n, f in stages.items():
            flush.fill_(2.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            f()
            e1.record(stream)
            times[n].append((e0, e1))
    torch.cuda.synchronize()
    assert moe.moe_read_status(bws) == moe.MOE_OK and moe.moe_read_status(rws) == moe.MOE_OK
    ms = {n: statistics.median(a.elapsed_time(bb) for a, bb in v) for n, v in times.items()}
    flops = 2.0 * synth.gemm_flops(w)  # dgrad + wgrad, each the forward GEMMs' flops
    recompute = synth.gemm_flops(w) * 2.0 / 3.0  # the gate/up GEMM run again
    peak = load_peaks()[0]["bf16_tflops"]  # measured burst: each call is timed alone
    tf = flops / (ms["grouped_mlp_backward"] / 1e3) / 1e12
    return {"metric": "MoE-layer bwd tokens/s", "value": round(T / (ms["backward"] / 1e3), 1), "unit": "tokens/s",
            "ms_per_step": round(ms["backward"], 4), "stages_ms": {n: round(v, 4) for n, v in ms.items() if n != "backward"},
            "grouped_gemm_tflops": round(tf, 1), "grouped_gemm_frac_of_peak": round(tf / peak, 3),
            "algorithmic_flops": flops, "recompute_flops": recompute,
            "router_flops": 4.0 * T * H * E,
            "training_step_ms": round(ms["forward_train"] + ms["backward"], 4),
            "training_step_graph_ms": round(ms["training_step_graph"], 4),
            "training_step_tokens_per_s": round(T / (ms["training_step_graph"] / 1e3), 1),
            "note": "the step: moe_backward_kept after moe_forward_train (gate/up pre-activations kept), with "
                    "training_step_graph: both replayed as one CUDA graph; "
                    "the router's backward and the auxiliary loss's gradient; backward_recompute reruns the gate/up "
                    "GEMM instead; grouped_gemm_tflops: dgrad + wgrad flops over the grouped MLP backward time "
                    "(which includes that recompute); router_flops: dW_router and dx's router share (tensor cores when E and H are multiples of "
                    "256, else fp32 SIMT); weight gradients "
                    "fp32; L2 flushed before each call"}


def set_gpu_local_affinity(dev):
    """Restricts this process to the CPUs local to the GPU (from sysfs, by its PCI bus id), so
    that pinned host buffers allocated now live on the GPU's host node. Returns (previous
    affinity, cpulist text), or (None, None) where that information is not available."""
    import torch
    try:
        props = torch.cuda.get_device_properties(dev)
        bus = "%04x:%02x:%02x.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
        with open("/sys/bus/pci/devices/%s/local_cpulist" % bus) as f:
            text = f.read().strip()
        cpus = set()
        for part in text.split(","):
            lo, _, hi = part.partition("-")
            cpus.update(range(int(lo), int(hi or lo) + 1))
        saved = os.sched_getaffinity(0)
        cpus &= saved
        if not cpus or cpus == saved:
            return None, None
        os.sched_setaffinity(0, cpus)
        return saved, text
    except (AttributeError, OSError, ValueError):
        return None, None


def launches_per_forward(w):
    # router logits, the routing (the library reports its launch count: one cooperative
    # launch, or the top-k launch and the scan), dispatch, 2 grouped GEMMs, combine
    import token_routing_expert_router_gb300 as moe
    cfg = moe.MoEConfig.make(**{kk: w[kk] for kk in (
        "T", "H", "E", "k", "F", "n_shared", "F_shared", "score_fn", "renorm", "n_groups",
        "topk_groups", "group_score", "routed_scale", "act_dtype", "xfer_dtype")})
    return 1 + moe.moe_route_launch_count(cfg) + 1 + 2 + 1


def cpu_baseline(w, n_tokens, seed=0):
    """The oracle as it stands, on n_tokens tokens of the workload (fp64, OpenMP)."""
    import oracle
    T, H, E, k, F = w["T"], w["H"], w["E"], w["k"], w["F"]
    qk = quant_kind(w)
    dt = synth.act_name(w)
    toks = np.arange(n_tokens)

    def qw(m):  # the oracle's own quantisation of a weight matrix
        if qk == 1:
            return oracle.dequant_blocks(*oracle.quant_blocks(m, 128, 128), 128, 128)
        return oracle.mx_dequant(*oracle.mx_quant(m)) if qk == 2 else m
    x = synth.rows(seed, synth.X, toks, H, 1.0, dt)
    wr = synth.normal(0, synth.W_ROUTER, (E, H), w["w_std"], dt)
    bias = synth.zipf_bias(0, E) if w["zipf"] else None
    t_or = 0.0
    t0 = time.perf_counter()
    logits = oracle.router_logits(x, wr, bias)
    sub = dict(w, T=n_tokens)
    idx, wt = oracle.route(logits, sub)
    counts, offsets, row_token, tok_row = oracle.permute(idx, E)
    if qk == 1:
        q, sc = oracle.quant_blocks(x, 1, 128)
        a = oracle.dequant_blocks(q, sc, 1, 128)
    elif qk == 2:
        a = oracle.mx_dequant(*oracle.mx_quant(x))
    else:
        a = x.astype(np.float64)
    xd = a[row_token]
    t_or += time.perf_counter() - t0
    yd = np.zeros((n_tokens * k, H))
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 == r0:
            continue
        g, u, d = synth.expert_weights(w, 0, e)  # drawing the weights is not timed
        t0 = time.perf_counter()
        g, u, d = qw(g), qw(u), qw(d)
        yd[r0:r1] = oracle.expert_mlp(xd[r0:r1], g, u, d, quant_h=qk)
        t_or += time.perf_counter() - t0
    ys = None
    if w["n_shared"]:
        Fs = w["F_shared"]
        g = synth.normal(0, synth.WS_GATE, (Fs, H), w["w_std"], dt)
        u = synth.normal(0, synth.WS_UP, (Fs, H), w["w_std"], dt)
        d = synth.normal(0, synth.WS_DOWN, (H, Fs), w["w_std"], dt)
        t0 = time.perf_counter()
        g, u, d = qw(g), qw(u), qw(d)
        ys = oracle.expert_mlp(a, g, u, d, quant_h=qk)
        t_or += time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.combine(yd, tok_row, wt, ys)
    t_or += time.perf_counter() - t0
    return {"value": round(n_tokens / t_or, 3), "unit": "tokens/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{n_tokens} tokens of the workload (router, top-k, permutation, every chosen expert's "
                      f"fp64 SwiGLU MLP, combine); OpenMP over rows; weight drawing not timed; "
                      f"{t_or:.1f} s of oracle time"}


def run_reference(args, w):
    world, rank, _ = rank_env()
    if rank != 0:
        return None  # the oracle runs once, on rank 0; the other ranks exit without work
    for _ in range(args.warmup):
        pass  # the oracle has no warm-up state; its build happens on import
    vals = []
    t_all = time.perf_counter()
    for i in range(args.steps):
        cb = cpu_baseline(w, args.cpu_tokens, seed=i)
        vals.append(cb)
    t_all = time.perf_counter() - t_all
    value = statistics.median(v["value"] for v in vals)
    cb = dict(vals[0])
    cb["value"] = value
    return {"impl": "reference", "metric": "MoE-layer fwd tokens/s", "value": value, "unit": "tokens/s",
            "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * t_all / args.steps, 1), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, world), "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-tokens", type=int, default=64)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="time direct moe_forward calls")
    ap.add_argument("--no-backward", action="store_true", help="skip the backward timing (bf16 layers)")
    ap.add_argument("--headline-only", action="store_true", help="skip the other layer shapes' entries")
    ap.add_argument("--tokens", type=int, default=0, help="override T (smaller profiling cases)")
    ap.add_argument("--experts", type=int, default=0, help="override E (smaller profiling cases)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    w = synth.WORKLOADS[args.workload]
    if args.tokens or args.experts:
        w = synth.scaled(w, T=args.tokens or w["T"], E=args.experts or w["E"],
                         name=f"{w['name']}_T{args.tokens or w['T']}_E{args.experts or w['E']}")
    line = run_reference(args, w) if args.impl == "reference" else run_gpu(args, w)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
