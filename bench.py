#!/usr/bin/env python
"""Benchmark of the MXFP4 MoE layer on GB300.

Headline workload: one gpt-oss-120b-shaped MoE layer in decode, T = 4 tokens,
H = I = 2880, E = 128, top-4 (bf16 hidden and router, MXFP4 experts, MXFP8
activations).  A step is one full forward of the layer (router, top-k, grouping,
gather, gate_up GEMM + SwiGLU + MXFP8, down GEMM, combine) through the C ABI.
Steps rotate over independently seeded layers whose packed weights (1.73 GB
each) together exceed L2 many times, so every step streams its experts from HBM.

The JSON line also carries the batched-decode (T = 32, skewed routing) and the
prefill (T = 2048) workloads, an end-to-end number with host buffers, the
roofline of the dominant kernel, the CPU oracle baseline and the SM clocks seen
during the timed region.  ``--impl reference`` times the CPU oracle instead.
Under torchrun every rank runs an independent replica (the layer needs no
collective); the value is the tokens of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import moe_synth as ms  # noqa: E402

METRIC = "MoE-layer tokens/s on 1 GB300; decode HBM GB/s, prefill TFLOPS vs peak"
H = I = 2880
E = 128
K_TOP = 4
# checkpoint-format bytes of one expert (packed E2M1 + E8M0 scales + bf16 bias)
GU_BYTES = 2 * I * (H // 2) + 2 * I * (H // 32) + 2 * I * 2
D_BYTES = H * (I // 2) + H * (I // 32) + H * 2
# NVFP4 weights: E4M3 block scales per 16 elements instead of E8M0 per 32
GU_BYTES_NV = 2 * I * (H // 2) + 2 * I * (H // 16) + 2 * I * 2
D_BYTES_NV = H * (I // 2) + H * (I // 16) + H * 2
FLOP_PER_ROW = 2 * (H * 2 * I + I * H)


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p.get("bf16_tflops_sustained", p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"moe_bench_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) >= 9:
                    rows.append(p)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        busy = sorted(sm)[len(sm) // 2:] if sm else []
        return {"sm_mhz": statistics.median(busy) if busy else None, "sm_max_mhz": max(mx) if mx else None,
                "samples": len(rows), "reasons": reasons}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        return dist, dist.get_rank(), ws, int(os.environ.get("LOCAL_RANK", "0"))
    return None, 0, 1, 0


def _max_over_ranks(dist, v: float, device) -> float:
    if dist is None:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _replica_tokens_per_s(world: int, T: int, ms_step: float) -> float:
    """Whole-job throughput of `world` independent replicas: the tokens of all
    ranks over the slowest rank's step time (already maxed over ranks)."""
    return world * T / (ms_step * 1e-3)


def _barrier(dist):
    if dist is not None:
        dist.barrier()


# ----------------------------------------------------------------------------- CPU oracle
def _oracle_tokens_per_s(T_sample: int, budget_s: float, seed: int = 0):
    """Single-threaded CPU oracle on the first tokens of the decode workload."""
    import oracle
    x = ms.make_tokens(seed, T_sample, H)
    rw, rb = ms.make_router(seed, H, E)
    _, ids, _ = oracle.route(x, rw, rb, K_TOP)
    need = sorted(set(ids.reshape(-1).tolist()))
    w = ms.make_expert_weights(seed, H, I, E, experts=need)
    full = []
    for t_sub in w:  # full-size arrays; experts not routed to stay zero and are never read
        z = torch.zeros((E,) + tuple(t_sub.shape[1:]), dtype=t_sub.dtype)
        z[need] = t_sub
        full.append(z)
    done, t0 = 0, time.perf_counter()
    while done < T_sample:
        oracle.moe_forward(x[done:done + 1], rw, rb, *full, k=K_TOP)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    el = time.perf_counter() - t0
    return done / el, done, el


def _oracle_tokens_per_s_all_cores(budget_s: float, seed: int = 0):
    """The same oracle, one token per task on every host core (it holds no global
    state, and its calls release the interpreter lock)."""
    import concurrent.futures as cf
    import oracle
    n = os.cpu_count() or 1
    T_sample = 2 * n
    x = ms.make_tokens(seed, T_sample, H)
    rw, rb = ms.make_router(seed, H, E)
    _, ids, _ = oracle.route(x, rw, rb, K_TOP)
    need = sorted(set(ids.reshape(-1).tolist()))
    w = ms.make_expert_weights(seed, H, I, E, experts=need)
    full = []
    for t_sub in w:
        z = torch.zeros((E,) + tuple(t_sub.shape[1:]), dtype=t_sub.dtype)
        z[need] = t_sub
        full.append(z)
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=n) as ex:
        list(ex.map(lambda t: oracle.moe_forward(x[t:t + 1], rw, rb, *full, k=K_TOP), range(T_sample)))
    el = time.perf_counter() - t0
    return T_sample / el, T_sample, el, n


def run_reference(args):
    dist, rank, world, _ = _dist()
    if rank != 0:
        return
    per_step = 1
    import oracle
    oracle.build()
    x = ms.make_tokens(0, args.warmup + args.steps, H)
    rw, rb = ms.make_router(0, H, E)
    _, ids, _ = oracle.route(x, rw, rb, K_TOP)
    need = sorted(set(ids.reshape(-1).tolist()))
    w = ms.make_expert_weights(0, H, I, E, experts=need)
    full = []
    for t_sub in w:
        z = torch.zeros((E,) + tuple(t_sub.shape[1:]), dtype=t_sub.dtype)
        z[need] = t_sub
        full.append(z)
    for i in range(args.warmup):
        oracle.moe_forward(x[i:i + 1], rw, rb, *full, k=K_TOP)
    t0 = time.perf_counter()
    for i in range(args.steps):
        j = args.warmup + i
        oracle.moe_forward(x[j:j + 1], rw, rb, *full, k=K_TOP)
    el = time.perf_counter() - t0
    v = args.steps * per_step / el
    line = {"metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": "decode_t4: gpt-oss-120b-shaped MoE layer, H=I=2880, E=128, top-4; "
                                   "each step one token of the workload through the CPU oracle"},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": f"{args.steps} tokens of the T=4 decode workload, one per step"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm
class Layers:
    """Independently seeded packed layers rotated through the steps."""

    def __init__(self, n: int, device, seed: int = 0, nvfp4: bool = False):
        import mxfp4_mixture_experts_gemv_gb300 as moe
        self.moe = moe
        self.dims = moe.LayerDims(E, H, I)
        self.packed, self.router = [], []
        for l in range(n):
            w = ms.make_expert_weights(seed, H, I, E, layer=l, device=device)
            self.packed.append(moe.pack_weights(self.dims, *w, nvfp4=nvfp4))
            torch.cuda.synchronize()
            del w
        self.n = n

    def routers(self, hot=0, hot_bias=0.0, device="cuda", seed=0):
        return [tuple(t.to(device) for t in ms.make_router(seed, H, E, layer=l, hot_experts=hot,
                                                            hot_bias=hot_bias)) for l in range(self.n)]


def _active_bytes(moe, ws, layout, n_active_out):
    cnt = moe.view(ws, layout.counts, (E,), torch.int32)
    n_active_out.append(int((cnt > 0).sum().item()))


def _workload(layers: Layers, T: int, hot: int, hot_bias: float, steps: int, warmup: int, device, dist,
              profile=True, seed=0, act_format="mxfp8"):
    """Time `steps` forwards of T tokens rotating over the layers; returns a stats dict."""
    moe = layers.moe
    routers = layers.routers(hot, hot_bias, device, seed)
    xs = [ms.make_tokens(seed, T, H, layer=l).to(device) for l in range(layers.n)]
    out = torch.empty((T, H), dtype=torch.bfloat16, device=device)
    ws = moe.alloc_workspace(layers.dims, T, K_TOP, device)
    layout = moe.workspace_layout(layers.dims, T, K_TOP)
    # routing statistics per layer (active experts -> algorithmic bytes)
    act = []
    for l in range(layers.n):
        moe.forward(layers.dims, xs[l], routers[l][0], routers[l][1], layers.packed[l], K_TOP, out=out, workspace=ws,
                    act_format=act_format)
        _active_bytes(moe, ws, layout, act)
    st = moe.device_status(ws)
    if st != moe.MOE_OK:
        raise RuntimeError(f"device status {moe.STATUS_NAMES.get(st, st)}: {moe.lib().moe_last_error().decode()}")
    # One CUDA graph per timed step, captured from the C-ABI call (the way a decode
    # loop runs it).
    for i in range(warmup):
        l = i % layers.n
        moe.forward(layers.dims, xs[l], routers[l][0], routers[l][1], layers.packed[l], K_TOP, out=out, workspace=ws,
                    act_format=act_format)
    torch.cuda.synchronize()

    def capture():
        graphs = []
        for i in range(steps):
            l = i % layers.n
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                moe.forward(layers.dims, xs[l], routers[l][0], routers[l][1], layers.packed[l], K_TOP, out=out,
                            workspace=ws, act_format=act_format)
            graphs.append(g)
        for i in range(min(warmup, steps)):
            graphs[i].replay()
        torch.cuda.synchronize()
        return graphs

    graphs = capture()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(dist)
    clocks = ClockSampler(torch.cuda.current_device())
    with clocks:
        e0.record(stream)
        for g in graphs:
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
    _barrier(dist)
    ms_total = e0.elapsed_time(e1)
    # per-step distribution (outside the timed region): each replay between its own events
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(graphs) + 1)]
    ev[0].record(stream)
    for i, g in enumerate(graphs):
        g.replay()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    per = sorted(ev[i].elapsed_time(ev[i + 1]) * 1e3 for i in range(len(graphs)))
    step_us = {"median": statistics.median(per), "min": per[0], "max": per[-1], "n": len(per),
               "note": "each replay between its own events, after the timed region"}
    del graphs
    # The per-stage split comes from a second set of graphs whose captures each
    # take one profiling slot (the stage events become graph nodes, so these
    # replays are not the timed ones).
    stage_ms, calls = {}, 0
    if profile:
        moe.profile_begin(steps)
        graphs = capture()
        for g in graphs:
            g.replay()
        torch.cuda.synchronize()
        stage_ms, calls = moe.profile_end()
        del graphs
    st = moe.device_status(ws)
    if st != moe.MOE_OK:
        raise RuntimeError(f"device status {moe.STATUS_NAMES.get(st, st)}")
    ms_step = _max_over_ranks(dist, ms_total / steps, device)
    seq = [act[i % layers.n] for i in range(steps)]
    n_act = sum(seq) / len(seq)
    gu_bytes = n_act * (GU_BYTES_NV if act_format == "nvfp4" else GU_BYTES)
    d_bytes = n_act * (D_BYTES_NV if act_format == "nvfp4" else D_BYTES)
    step_bytes = gu_bytes + d_bytes + E * H * 2 + E * 2 + 2 * T * H * 2
    flop = T * K_TOP * FLOP_PER_ROW + 2 * T * E * H
    stage_avg = {k: v / max(calls, 1) for k, v in stage_ms.items()}
    return dict(T=T, ms_per_step=ms_step, tokens_per_s=T / (ms_step * 1e-3), active_experts=n_act,
                step_bytes=step_bytes, gu_bytes=gu_bytes, d_bytes=d_bytes, flop=flop,
                gbs=step_bytes / (ms_step * 1e-3) / 1e9, tflops=flop / (ms_step * 1e-3) / 1e12,
                stage_ms=stage_avg, clocks=clocks.summary(), xs=xs, routers=routers, out=out, ws=ws,
                step_us=step_us)


def _stack(layers: Layers, n_layers: int, T: int, steps: int, warmup: int, device, dist, graph: bool,
           act_format="mxfp8"):
    """x <- x + moe(rmsnorm(x)) over n_layers independently seeded layers (all resident)."""
    moe = layers.moe
    while len(layers.packed) < n_layers:
        w = ms.make_expert_weights(0, H, I, E, layer=len(layers.packed), device=device)
        layers.packed.append(moe.pack_weights(layers.dims, *w))
        torch.cuda.synchronize()
        del w
    routers = [tuple(t.to(device) for t in ms.make_router(0, H, E, layer=l)) for l in range(n_layers)]
    x0 = ms.make_tokens(0, T, H).to(device).float()
    x_res = torch.empty_like(x0)
    hidden = torch.empty((T, H), dtype=torch.bfloat16, device=device)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=device)
    ws = moe.alloc_workspace(layers.dims, T, K_TOP, device)
    lay = moe.workspace_layout(layers.dims, T, K_TOP)

    def step(count=None):
        x_res.copy_(x0)
        prev = None
        for l in range(n_layers):
            moe.residual_rmsnorm(x_res, prev, hidden)
            moe.forward(layers.dims, hidden, routers[l][0], routers[l][1], layers.packed[l], K_TOP, out=out,
                        workspace=ws, act_format=act_format)
            if count is not None:
                count.append(int((moe.view(ws, lay.counts, (E,), torch.int32) > 0).sum().item()))
            prev = out
        moe.residual_rmsnorm(x_res, out, hidden)

    act = []
    step(act)  # also the active experts of every layer
    st = moe.device_status(ws)
    if st != moe.MOE_OK:
        raise RuntimeError(f"stack: device status {moe.STATUS_NAMES.get(st, st)}")
    g = None
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
    run = g.replay if g is not None else step
    for _ in range(warmup):
        run()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    _barrier(dist)
    clocks = ClockSampler(torch.cuda.current_device())
    with clocks:
        e0.record(stream)
        for _ in range(steps):
            run()
        e1.record(stream)
        torch.cuda.synchronize()
    _barrier(dist)
    ms_step = _max_over_ranks(dist, e0.elapsed_time(e1) / steps, device)
    step_bytes = sum(a * (GU_BYTES + D_BYTES) for a in act) + n_layers * (E * H * 2 + E * 2 + 2 * T * H * 2)
    flop = n_layers * (T * K_TOP * FLOP_PER_ROW + 2 * T * E * H)
    return {"T": T, "layers": n_layers, "tokens_per_s": T / (ms_step * 1e-3), "ms_per_step": ms_step,
            "ms_per_layer": ms_step / n_layers, "active_experts_per_layer": sum(act) / len(act),
            "algorithmic_bytes": step_bytes, "gbs": step_bytes / (ms_step * 1e-3) / 1e9,
            "tflops": flop / (ms_step * 1e-3) / 1e12, "timing": "CUDA graph of the whole step" if graph else
            "stream of C-ABI calls", "clocks": clocks.summary()}


def _dense(N: int, K: int, T: int, steps: int, warmup: int, device, hbm_peak: float, fp8_peak: float):
    """One dense MXFP4 linear (bf16 weights of the given shape quantised on the device)
    at T tokens: the default path, and for T <= 4 both forced paths.  Enough weight
    copies rotate through the steps to exceed L2; each step is one graph replay."""
    import mxfp4_mixture_experts_gemv_gb300 as moe
    copies = max(1, -(-(256 << 20) // (N * K // 2)))
    packs = []
    for c in range(copies):
        g = torch.Generator(device=device).manual_seed(1000 + c)
        wt = (torch.randn(N, K, generator=g, device=device) * 0.05).to(torch.bfloat16)
        b = (torch.randn(N, generator=g, device=device) * 0.02).to(torch.bfloat16)
        packs.append(moe.dense_pack(*moe.dense_quantize_weights(wt), b))
        del wt
    x = ms.make_tokens(7, T, K).to(device)
    out = torch.empty((T, N), dtype=torch.bfloat16, device=device)
    ws = moe._alloc_aligned(max(moe.lib().moe_dense_workspace_size(N, K, T), 256), device)
    res = {"N": N, "K": K, "T": T, "weight_copies_rotated": copies}
    wbytes = N * (K // 2) + N * (K // 32) + N * 4
    step_bytes = wbytes + T * K * 2 + T * N * 2
    for path in (["auto", "cuda_cores", "weights_m"] if T <= 4 else ["auto"]):
        moe.set_plan(0, "auto", path)
        try:
            for i in range(warmup):
                moe.dense_forward(N, K, x, packs[i % copies], out=out, workspace=ws)
            graphs = []
            for i in range(steps):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    moe.dense_forward(N, K, x, packs[i % copies], out=out, workspace=ws)
                graphs.append(g)
            torch.cuda.synchronize()
            stream = torch.cuda.current_stream()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for g in graphs:
                g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / steps
            del graphs
        finally:
            moe.set_plan(0, "auto")
        res[path] = {"us_per_call": us, "gbs": step_bytes / (us * 1e-6) / 1e9,
                     "hbm_frac": step_bytes / (us * 1e-6) / 1e9 / hbm_peak,
                     "tflops": 2.0 * T * N * K / (us * 1e-6) / 1e12,
                     "tflops_frac_of_fp8_peak": 2.0 * T * N * K / (us * 1e-6) / 1e12 / fp8_peak}
    res["algorithmic_bytes"] = step_bytes
    del packs
    torch.cuda.empty_cache()
    return res


def _e2e(layers: Layers, w: dict, steps: int, warmup: int, device, dist):
    """Same workload through the C ABI with pinned host buffers: H2D of x and D2H of out each step."""
    moe = layers.moe
    T = w["T"]
    hx = [x.cpu().pin_memory() for x in w["xs"]]
    hout = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    dx = torch.empty((T, H), dtype=torch.bfloat16, device=device)
    out, ws, routers = w["out"], w["ws"], w["routers"]
    stream = torch.cuda.current_stream()

    def step(i):
        l = i % layers.n
        dx.copy_(hx[l], non_blocking=True)
        moe.forward(layers.dims, dx, routers[l][0], routers[l][1], layers.packed[l], K_TOP, out=out, workspace=ws)
        hout.copy_(out, non_blocking=True)

    for i in range(warmup):
        step(i)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    _barrier(dist)
    e0.record(stream)
    for i in range(steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    _barrier(dist)
    ms_step = _max_over_ranks(dist, e0.elapsed_time(e1) / steps, device)
    # the same step (H2D of x, forward, D2H of out) captured into one graph per layer
    gs = []
    for l in range(layers.n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(l)
        gs.append(g)
    for i in range(warmup):
        gs[i % layers.n].replay()
    torch.cuda.synchronize()
    _barrier(dist)
    e0.record(stream)
    for i in range(steps):
        gs[i % layers.n].replay()
    e1.record(stream)
    torch.cuda.synchronize()
    _barrier(dist)
    ms_graph = _max_over_ranks(dist, e0.elapsed_time(e1) / steps, device)
    # two requests in flight: steps alternate between two streams, each with its own
    # input, output, workspace and pinned host buffers, so one step's copies overlap
    # the other's kernels; every step still pays its own H2D and D2H
    streams = [torch.cuda.Stream(device=device) for _ in range(2)]
    bufs = [(dx, out, ws, hout)]
    bufs.append((torch.empty_like(dx), torch.empty_like(out), moe.alloc_workspace(layers.dims, T, K_TOP, device),
                 torch.empty_like(hout).pin_memory()))

    def step2(i):
        l = i % layers.n
        dxi, outi, wsi, houti = bufs[i % 2]
        with torch.cuda.stream(streams[i % 2]):
            dxi.copy_(hx[l], non_blocking=True)
            moe.forward(layers.dims, dxi, routers[l][0], routers[l][1], layers.packed[l], K_TOP, out=outi,
                        workspace=wsi)
            houti.copy_(outi, non_blocking=True)

    torch.cuda.synchronize()
    for i in range(warmup):
        step2(i)
    torch.cuda.synchronize()
    _barrier(dist)
    e0.record(stream)
    for st in streams:
        st.wait_event(e0)
    for i in range(steps):
        step2(i)
    for st in streams:
        stream.wait_stream(st)
    e1.record(stream)
    torch.cuda.synchronize()
    _barrier(dist)
    ms_pipe = _max_over_ranks(dist, e0.elapsed_time(e1) / steps, device)
    return {"value": T / (ms_step * 1e-3), "unit": "tokens/s", "ms_per_step": ms_step,
            "h2d_bytes_per_step": T * H * 2, "d2h_bytes_per_step": T * H * 2,
            "api": "moe_forward per step from Python, pinned host x in / out",
            "graph": {"value": T / (ms_graph * 1e-3), "ms_per_step": ms_graph,
                      "api": "the same step captured into a CUDA graph per layer"},
            "pipelined": {"value": T / (ms_pipe * 1e-3), "ms_per_step": ms_pipe,
                          "api": "the same per-step calls with two requests in flight on two streams "
                                 "(own buffers and workspace each); copies overlap the other request's kernels"}}


def _source_hash(names) -> str:
    """First 16 hex digits of the SHA-256 of the named kernel sources, concatenated."""
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "mxfp4_mixture_experts_gemv_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's sources
    (the kernel file and the headers it includes) are unchanged."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[f"{kernel}@{workload}"]
        if _source_hash(rec["sources"]) != rec["sources_sha256_16"]:
            return None
        return rec["dram_bytes_per_launch"]
    except Exception:
        return None


def run_ours(args):
    dist, rank, world, local = _dist()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import mxfp4_mixture_experts_gemv_gb300 as moe
    if not os.path.exists(moe.LIB_PATH):
        from mxfp4_mixture_experts_gemv_gb300 import build as b
        b.build()
    moe.lib()
    hbm_peak, bf16_peak, bf16_sust, peak_src = _peaks()
    fp8_peak = 2 * bf16_peak  # kind::mxf8f6f4 runs at the fp8 rate: 2x the bf16 dense rate (nominal ratio)
    fp4_peak = 6 * bf16_peak  # kind::mxf4: the dense fp4 rate, 13.5 / 2.25 times the bf16 rate (nominal ratio)
    t_gen = time.perf_counter()
    layers = Layers(args.layers, device)
    t_gen = time.perf_counter() - t_gen

    main = _workload(layers, 4, 0, 0.0, args.steps, args.warmup, device, dist)
    e2e = _e2e(layers, main, args.steps, args.warmup, device, dist)
    extra = {}
    if not args.no_extra:
        for name, T, hot, hb, n in (("decode_t32_skewed", 32, 16, 1.0, args.steps),
                                    ("prefill_t2048", 2048, 0, 0.0, max(10, args.steps // 5))):
            w = _workload(layers, T, hot, hb, n, min(args.warmup, 3), device, dist)
            mlp_ms = w["stage_ms"].get("expert_mlp", 0) or float("nan")
            expert_flop = T * K_TOP * FLOP_PER_ROW
            extra[name] = {
                "T": T, "tokens_per_s": _replica_tokens_per_s(world, T, w["ms_per_step"]),
                "ms_per_step": w["ms_per_step"],
                "active_experts": w["active_experts"], "algorithmic_bytes": w["step_bytes"],
                "gbs": w["gbs"], "tflops": w["tflops"],
                "expert_mlp_gbs": (w["gu_bytes"] + w["d_bytes"]) / (mlp_ms * 1e-3) / 1e9,
                "expert_mlp_tflops": expert_flop / (mlp_ms * 1e-3) / 1e12,
                "expert_mlp_tflops_frac_of_fp8_peak": expert_flop / (mlp_ms * 1e-3) / 1e12 / fp8_peak,
                "stage_ms": w["stage_ms"], "clocks": w["clocks"]}
            del w

    if not args.no_extra:
        # the FP4 x FP4 variant (activations in MXFP4, tcgen05 kind::mxf4)
        for name, T, n in (("mxfp4act_decode_t4", 4, args.steps), ("mxfp4act_prefill_t2048", 2048, max(10, args.steps // 5))):
            w = _workload(layers, T, 0, 0.0, n, min(args.warmup, 3), device, dist, act_format="mxfp4")
            mlp_ms = w["stage_ms"].get("expert_mlp", 0) or float("nan")
            expert_flop = T * K_TOP * FLOP_PER_ROW
            extra[name] = {
                "T": T, "act_format": "mxfp4", "tokens_per_s": _replica_tokens_per_s(world, T, w["ms_per_step"]),
                "ms_per_step": w["ms_per_step"], "active_experts": w["active_experts"],
                "algorithmic_bytes": w["step_bytes"], "gbs": w["gbs"], "hbm_frac": w["gbs"] / hbm_peak,
                "tflops": w["tflops"],
                "expert_mlp_gbs": (w["gu_bytes"] + w["d_bytes"]) / (mlp_ms * 1e-3) / 1e9,
                "expert_mlp_tflops": expert_flop / (mlp_ms * 1e-3) / 1e12,
                "expert_mlp_tflops_frac_of_fp4_peak": expert_flop / (mlp_ms * 1e-3) / 1e12 / fp4_peak,
                "stage_ms": w["stage_ms"], "clocks": w["clocks"]}
            del w

    if not args.no_extra:
        # the NVFP4 variant: the MXFP4 layers converted to NVFP4 while packing, NVFP4
        # activations (tcgen05 kind::mxf4nvf4)
        nv_layers = Layers(args.layers, device, nvfp4=True)
        for name, T, n in (("nvfp4_decode_t4", 4, args.steps), ("nvfp4_prefill_t2048", 2048, max(10, args.steps // 5))):
            w = _workload(nv_layers, T, 0, 0.0, n, min(args.warmup, 3), device, dist, act_format="nvfp4")
            mlp_ms = w["stage_ms"].get("expert_mlp", 0) or float("nan")
            expert_flop = T * K_TOP * FLOP_PER_ROW
            extra[name] = {
                "T": T, "act_format": "nvfp4", "tokens_per_s": _replica_tokens_per_s(world, T, w["ms_per_step"]),
                "ms_per_step": w["ms_per_step"], "active_experts": w["active_experts"],
                "algorithmic_bytes": w["step_bytes"], "gbs": w["gbs"], "hbm_frac": w["gbs"] / hbm_peak,
                "tflops": w["tflops"],
                "expert_mlp_gbs": (w["gu_bytes"] + w["d_bytes"]) / (mlp_ms * 1e-3) / 1e9,
                "expert_mlp_tflops": expert_flop / (mlp_ms * 1e-3) / 1e12,
                "expert_mlp_tflops_frac_of_fp4_peak": expert_flop / (mlp_ms * 1e-3) / 1e12 / fp4_peak,
                "stage_ms": w["stage_ms"], "clocks": w["clocks"]}
            del w
        del nv_layers
        torch.cuda.empty_cache()
        # dense MXFP4 linears of the same model: attention projections and LM head
        for name, N, K, T in (("dense_qkv_t4", 5120, 2880, 4), ("dense_o_t4", 2880, 4096, 4),
                              ("dense_lm_head_t1", 201088, 2880, 1), ("dense_qkv_t2048", 5120, 2880, 2048)):
            extra[name] = _dense(N, K, T, args.steps, min(args.warmup, 3), device, hbm_peak, fp8_peak)

    if not args.no_extra and not args.no_stack:
        n_l = 36
        pre = _stack(layers, n_l, 8192, 2, 1, device, dist, graph=False)
        pre["tflops_frac_of_fp8_peak"] = pre["tflops"] / fp8_peak
        extra["stack36_prefill_t8192"] = pre
        dec = _stack(layers, n_l, 4, max(5, args.steps // 5), 2, device, dist, graph=True)
        dec["hbm_frac"] = dec["gbs"] / hbm_peak
        extra["stack36_decode_t4"] = dec
        pre4 = _stack(layers, n_l, 8192, 2, 1, device, dist, graph=False, act_format="mxfp4")
        pre4["tflops_frac_of_fp4_peak"] = pre4["tflops"] / fp4_peak
        pre4["tflops_frac_of_fp8_peak"] = pre4["tflops"] / fp8_peak
        pre4["act_format"] = "mxfp4"
        extra["mxfp4act_stack36_prefill_t8192"] = pre4

    cpu_v, cpu_n, cpu_s = (None, 0, 0.0)
    cpu_all = None
    if rank == 0 and not args.no_cpu:
        cpu_v, cpu_n, cpu_s = _oracle_tokens_per_s(64, args.cpu_budget)
        av, an, asec, acores = _oracle_tokens_per_s_all_cores(args.cpu_budget)
        cpu_all = {"value": av, "unit": "tokens/s", "cores": acores, "kind": "oracle",
                   "sample": f"{an} tokens of the decode workload, one per task on {acores} threads "
                             f"({asec:.1f} s, fp64)"}

    mlp_ms = main["stage_ms"].get("expert_mlp", 0.0)
    mlp_bytes = main["gu_bytes"] + main["d_bytes"]
    achieved = mlp_bytes / (mlp_ms * 1e-3) / 1e9 if mlp_ms else None
    value = _replica_tokens_per_s(world, main["T"], main["ms_per_step"])
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": main["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 x e2m1 block-scaled (E8M0), fp32 accumulate", "data": "synthetic",
        "config": {"workload": "decode_t4: one gpt-oss-120b-shaped MoE layer, T=4 tokens, H=I=2880, E=128, "
                               "top-4, bf16 hidden/router, MXFP4 experts, MXFP8 activations",
                   "layers_rotated": args.layers,
                   "timing": "one CUDA graph per step captured from moe_forward, CUDA events around the replays",
                   "l2": f"inputs larger than L2: {args.layers} independently seeded layers "
                         f"({args.layers * moe.packed_size(layers.dims) / 1e9:.1f} GB packed) rotated per step",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "decode_hbm_gbs": main["gbs"], "decode_hbm_frac": main["gbs"] / hbm_peak,
        "active_experts_per_step": main["active_experts"],
        "roofline": {"kernel": "expert_mlp_kernel (gate_up + down + combine, tcgen05 kind::mxf8f6f4)",
                     "bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": (achieved / hbm_peak) if achieved else None,
                     "traffic": _traffic("expert_mlp_kernel", "decode_t4"),
                     "algorithmic_bytes_per_launch": mlp_bytes,
                     "peak_source": f"{peak_src} hbm_gbs (copy)"},
        "stage_ms": main["stage_ms"],
        "e2e": e2e,
        "gpu_launches": args.steps * 2,
        "gpu_launches_note": "per step: the fused routing kernel and the expert kernel (T <= 32)",
        "clocks": main["clocks"],
        "cpu_baseline": ({"value": cpu_v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                          "sample": f"{cpu_n} tokens of the decode workload ({cpu_s:.1f} s, single-threaded fp64)"}
                         if cpu_v else None),
        "cpu_baseline_all_cores": cpu_all,
        "step_us_distribution": main["step_us"],
        "workloads": extra,
        "peaks": {"hbm_gbs": hbm_peak, "fp8_tflops": fp8_peak, "fp4_tflops": fp4_peak, "source": peak_src},
        "setup_s": t_gen,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_case(T: int, calls: int, plan=None, act_format: str = "mxfp8"):
    """A small profiling target: one layer (about 2.3 GB of packed weights on the
    device), ``calls`` forward calls on the default stream, then the device status."""
    import torch
    import moe_synth as ms
    import mxfp4_mixture_experts_gemv_gb300 as moe
    H = I = 2880
    E, k = 128, 4
    dims = moe.LayerDims(E, H, I)
    w = ms.make_expert_weights(0, H, I, E, device="cuda")
    packed = moe.pack_weights(dims, *w)
    del w
    rw, rb = [t.cuda() for t in ms.make_router(0, H, E, hot_experts=16 if T == 32 else 0, hot_bias=1.0)]
    x = ms.make_tokens(0, T, H).cuda()
    if plan:
        moe.set_plan(int(plan[0]), plan[1], plan[2])
    ws = moe.alloc_workspace(dims, T, k)
    for _ in range(calls):
        moe.forward(dims, x, rw, rb, packed, k, workspace=ws, act_format=act_format)
    torch.cuda.synchronize()
    st = moe.device_status(ws)
    print(f"case T={T} plan={plan} act={act_format}: {calls} calls, device status {st}", flush=True)
    if st != 0:
        raise SystemExit(1)


SWEEP_T = (1, 2, 4, 8, 12, 16, 24, 32, 48, 64, 96, 128, 256, 512, 1024, 2048, 4096, 8192)


def _plans_for(T: int):
    """Candidate (tile_rows, routing path, expert kernel) for T tokens: every tile
    height the kernels have, every routing path whose capacity covers T, and both
    expert kernels on 128-row tiles."""
    routes = (["cluster"] if T <= 8 else []) + (["grid"] if T <= 32 else []) + ["tensor_core"]
    rows = (8, 16, 32, 64, 128) if T <= 256 else (32, 64, 128)
    out = []
    for r in rows:
        for rt in routes:
            for ex in (("weights_m", "tokens_m") if r == 128 else ("auto",)):
                out.append((r, rt, ex))
    return out


def run_sweep(args):
    """Plan sweep: for each T, the median step time of every candidate plan
    (moe_set_plan) on the gpt-oss-shaped layer, layers rotated so that weights
    stream from HBM; one JSON line per (T, plan), then the table of the fastest."""
    import mxfp4_mixture_experts_gemv_gb300 as moe
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    if not os.path.exists(moe.LIB_PATH):
        from mxfp4_mixture_experts_gemv_gb300 import build as b
        b.build()
    layers = Layers(args.layers, device)
    routers = layers.routers(device=device)
    best = {}
    for T in (args.sweep_t or SWEEP_T):
        xs = [ms.make_tokens(0, T, H, layer=l).to(device) for l in range(layers.n)]
        out = torch.empty((T, H), dtype=torch.bfloat16, device=device)
        rows = []
        for tr, rt, ex in _plans_for(T):
            moe.set_plan(tr, rt, ex)
            try:
                ws = moe.alloc_workspace(layers.dims, T, K_TOP, device)
                for l in range(layers.n):  # warm-up, and the plan must run
                    moe.forward(layers.dims, xs[l], routers[l][0], routers[l][1], layers.packed[l], K_TOP, out=out,
                                workspace=ws, act_format=args.act)
                st = moe.device_status(ws)
                if st != moe.MOE_OK:
                    raise RuntimeError(f"device status {st}")
                graphs = []
                for i in range(args.steps):
                    l = i % layers.n
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g):
                        moe.forward(layers.dims, xs[l], routers[l][0], routers[l][1], layers.packed[l], K_TOP,
                                    out=out, workspace=ws, act_format=args.act)
                    graphs.append(g)
                for g in graphs[:args.warmup]:
                    g.replay()
                torch.cuda.synchronize()
                stream = torch.cuda.current_stream()
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(graphs) + 1)]
                ev[0].record(stream)
                for i, g in enumerate(graphs):
                    g.replay()
                    ev[i + 1].record(stream)
                torch.cuda.synchronize()
                us = statistics.median(ev[i].elapsed_time(ev[i + 1]) * 1e3 for i in range(len(graphs)))
                del graphs, ws
            finally:
                moe.set_plan(0, "auto")
            line = {"sweep": "plan", "act": args.act, "T": T, "tile_rows": tr, "route": rt, "expert": ex, "step_us": us,
                    "tokens_per_s": T / (us * 1e-6)}
            rows.append(line)
            print(json.dumps(line), flush=True)
        # the automatic plan, for comparison
        ws = moe.alloc_workspace(layers.dims, T, K_TOP, device)
        lay = moe.workspace_layout(layers.dims, T, K_TOP, args.act)
        fastest = min(rows, key=lambda r: r["step_us"])
        best[T] = {"fastest": (fastest["tile_rows"], fastest["route"], fastest["expert"], round(fastest["step_us"], 1)),
                   "auto_tile_rows": lay.tile_rows}
        del ws
    print(json.dumps({"sweep": "summary", "best": best}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=8, help="independently seeded layers rotated per step")
    ap.add_argument("--no-extra", action="store_true", help="only the headline decode workload")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-stack", action="store_true", help="skip the 36-layer stack workloads")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of CPU oracle work")
    ap.add_argument("--sweep", action="store_true",
                    help="plan sweep: median step time of every tile-height and routing-path candidate per T")
    ap.add_argument("--sweep-t", type=int, nargs="*", default=None, help="token counts of the plan sweep")
    ap.add_argument("--plan", nargs=3, default=None, metavar=("TILE_ROWS", "ROUTE", "EXPERT"),
                    help="with --case: force a plan (tile rows, routing path, expert kernel)")
    ap.add_argument("--act", default="mxfp8", choices=["mxfp8", "mxfp4"],
                    help="with --case or --sweep: activation format")
    ap.add_argument("--case", type=int, default=None, metavar="T",
                    help="profiling run: one gpt-oss-shaped layer at T tokens, warmup + steps plain "
                         "forward calls, no timing and no JSON line (T=32 uses the skewed router)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.case is not None:
        run_case(args.case, args.warmup + args.steps, args.plan, args.act)
    elif args.sweep:
        run_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
