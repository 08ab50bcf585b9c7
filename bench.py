"""Benchmark of the fused decode MoE layer: us per layer launch and achieved
HBM GB/s against the byte roofline, one JSON line on stdout.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload dsv3_t1|dsv3_t8|dsv3_t64] [--no-sweep] [--sweep-wide]

A step is one launch of the whole layer (group table, gate/up + SwiGLU,
down, router weights, shared expert, residual, bf16 write) over one batch.
The default workload is the DeepSeek-V3-shaped decode layer at T=1 (H=7168,
routed I=2048 NVFP4 E=256 top-8, shared I=2048 FP8 128x128 blocks, uniform
routing). Four copies of the layer's weights are resident and the steps
rotate over them, so each step reads weights that are not in L2 (126 MB).
Every timing is also taken with the launches captured in a CUDA graph and
replayed (`graph_us_per_launch`), and in `chain` the same launches back to back
in four forms, alternating within every round: plain, chained (MOE_FLAG_CHAIN:
each may start under the previous one), with the next layer's first
shared-expert stages brought into L2 during each launch's tail
(moe_fused_decode_next), and both. The T=8 and T=64 workloads are timed too, under `sweep`
with the T=8 and T=64 layers again under the opt-in FP8 intermediate blocks
(--no-sweep skips them); --sweep-wide adds the wide-expert layer (E=384 top-8, uniform routing) at
T = 1, 2, 4, ..., 256 with 4 distinct layers' weights resident, run back to
back, plain and chained. --impl reference times the fp64 CPU oracle on whole launches of the
same workload (the reference arm). Under torchrun every rank runs its own replica
(the build has no cross-GPU exchange); rank 0 prints the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOADS = {
    "dsv3_t1": dict(T=1, routing="uniform"),
    "dsv3_t8": dict(T=8, routing="mtp"),
    "dsv3_t64": dict(T=64, routing="zipf"),
}
# sweep points beyond the metric's workloads: the T=1 layer with the router
# (bf16 [E][H] gate, bf16 correction bias, top-8, renormalised, scale 2.5)
# computed inside the same launch
ROUTED = {"dsv3_t1_routed": dict(T=1)}
# the opt-in FP8 intermediate blocks (MOE_FLAG_FP8_MID) on the workloads above
FP8_MID = {"dsv3_t8_fp8mid": "dsv3_t8", "dsv3_t64_fp8mid": "dsv3_t64"}
N_COPIES = 4
HEAD_START_CYCLES = 4_000_000  # device sleep (about 2 ms) before a back-to-back timed region
KERNEL_SOURCES = ["moe_layer_decode_persistent_b300/csrc/api.cu",
                  "moe_layer_decode_persistent_b300/csrc/fused_fma.cuh",
                  "moe_layer_decode_persistent_b300/csrc/fused_tc.cuh",
                  "moe_layer_decode_persistent_b300/csrc/sm100.cuh",
                  "moe_layer_decode_persistent_b300/csrc/group_table.cuh",
                  "moe_layer_decode_persistent_b300/csrc/moe_common.cuh",
                  "moe_layer_decode_persistent_b300/csrc/router.cuh"]


def _code_only(text: str) -> str:
    """C/C++ source without comments and with whitespace collapsed, so that a
    change of comments alone does not count as a change of the kernel."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif c in "\"'":  # string or character literal, copied as is
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash() -> str:
    """Hash of the kernel sources' code (comments and whitespace ignored)."""
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        fp = os.path.join(ROOT, p)
        if os.path.exists(fp):
            h.update(_code_only(open(fp, encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6400.0, "fallback"


def traffic_record(kernel: str):
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    rec = d.get(kernel)
    if not rec or rec.get("source_hash") != kernel_source_hash():
        return None
    return rec


class ClockSampler:
    """nvidia-smi SM clock / throttle sampling during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [v.strip() for v in ln.split(",")]
            if len(f) < 6:
                continue
            try:
                sm.append(float(f[0]))
                mx = max(mx, float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[2:6]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int, device=None) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def algorithmic_bytes(layer, ids) -> tuple[int, int]:
    T, H, K = layer.shape.T, layer.shape.H, layer.shape.K
    distinct = len(set(int(e) for e in ids.reshape(-1).tolist() if 0 <= int(e) < layer.shape.E))
    b = distinct * layer.routed.nbytes_expert() + layer.shared.nbytes_expert() + 2 * T * H * 2 + T * K * 8
    return b, distinct


def run_ours(args, rank, world, local):
    import torch

    from moe_layer_decode_persistent_b300 import binding as B
    from moe_layer_decode_persistent_b300 import build, inputs

    build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = WORKLOADS[args.workload]
    shape = inputs.dsv3(wl["T"], E=args.experts)
    L = inputs.make_layer(shape, wl["routing"], 0, dev, inputs.FMT_NVFP4, inputs.FMT_FP8_B128)
    copies = [(L.routed, L.shared)]
    for _ in range(args.copies - 1):
        r = inputs.ExpertSet(**{k: (v.clone() if isinstance(v, torch.Tensor) else v)
                                for k, v in L.routed.__dict__.items()})
        s = inputs.ExpertSet(**{k: (v.clone() if isinstance(v, torch.Tensor) else v)
                                for k, v in L.shared.__dict__.items()})
        copies.append((r, s))
    weights = [(B.make_weights(r), B.make_weights(s)) for r, s in copies]
    sh = B.make_shape(shape.T, shape.H, shape.I, shape.I_shared, shape.E, shape.K, args.flags)
    ws = torch.empty(B.moe_workspace_bytes_host(sh), dtype=torch.uint8, device=dev)
    B.moe_workspace_init(ws)
    out = torch.empty(shape.T, shape.H, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    algo_bytes, distinct = algorithmic_bytes(L, L.topk_ids.cpu())

    def launch(i):
        rw, sw = weights[i % len(weights)]
        B.moe_fused_decode(L.x, L.topk_ids, L.topk_w, rw, sw, out, sh, ws, stream=stream)

    # End to end through the host-buffer entry point (pinned buffers, copies
    # inside), before the clock sampler has ever run in this process: once
    # nvidia-smi has run, this synchronous loop measured 151 us a step
    # instead of 97 us for the rest of the process.
    e2e_us = None
    if not args.no_e2e:
        xh = L.x.cpu().pin_memory()
        ih = L.topk_ids.cpu().pin_memory()
        wh = L.topk_w.cpu().pin_memory()
        oh = torch.empty_like(xh).pin_memory()

        def launch_host(i):
            rw, sw = weights[i % len(weights)]
            B.moe_fused_decode_host(xh, ih, wh, rw, sw, oh, sh, ws, stream=stream)

        for i in range(max(3, args.warmup)):
            launch_host(i)
        barrier(world)
        h0 = time.perf_counter()
        for i in range(args.steps):
            launch_host(i)
        e2e_us = (time.perf_counter() - h0) / args.steps * 1e6
        e2e_us = max_over_ranks(e2e_us, world, dev)
        launch(0)  # the device entry on the same inputs gives the same bits
        torch.cuda.synchronize()
        assert torch.equal(oh.view(torch.int16), out.cpu().view(torch.int16))

    # the clock sampler starts before the warm-up (its start-up pause would
    # otherwise leave the GPU idle right before the timed region) and stops
    # after the device-timed launches; a second sampler covers the graph,
    # chained and sweep timings
    clk = ClockSampler(local).__enter__()
    for i in range(args.warmup):
        launch(i)
    torch.cuda.synchronize()
    assert B.moe_read_error(ws) == 0

    # the timed region: K launches back to back between two events (a short
    # device-side sleep ahead of the first event lets the host queue launches
    # before the clock starts, so host launch latency does not open gaps)
    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(HEAD_START_CYCLES)
    t0.record(stream)
    for i in range(args.steps):
        launch(i)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    err = B.moe_read_error(ws)
    total_ms = t0.elapsed_time(t1)
    ms_per_step = max_over_ranks(total_ms / args.steps, world, dev)
    us_launch_max = ms_per_step * 1e3

    # the same launches once more with an event pair around each, for the
    # spread of single launches (events between launches add their own gaps)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for i in range(args.steps):
        starts[i].record(stream)
        launch(i)
        ends[i].record(stream)
    torch.cuda.synchronize()
    per_launch = [s.elapsed_time(e) * 1e3 for s, e in zip(starts, ends)]  # us
    clk.__exit__()

    # end to end through the host-buffer entry point (pinned buffers, copies inside)
    if args.no_e2e:
        del copies, weights
        torch.cuda.empty_cache()
        clk2 = ClockSampler(local).__enter__()
        wide = wide_sweep(args, dev) if args.sweep_wide else {}
        clk2.__exit__()
        return dict(us_launch=us_launch_max, ms_per_step=ms_per_step, algo_bytes=algo_bytes,
                    distinct=distinct, clocks=clk.summary(), err=err, e2e_us=None, h2d=0, d2h=0,
                    sweep={}, wide=wide, graph_us=None, T=shape.T, per_launch=per_launch, chain=None,
                    clocks_after=clk2.summary() if args.sweep_wide else None)
    clk2 = ClockSampler(local).__enter__()

    def launch_s(i, s):
        rw, sw = weights[i % len(weights)]
        B.moe_fused_decode(L.x, L.topk_ids, L.topk_w, rw, sw, out, sh, ws, stream=s)

    graph_us = graph_us_per_launch(launch_s, 4 * len(weights))
    assert B.moe_read_error(ws) == 0

    # the same layers back to back in three more forms, alternating with the
    # plain launches: chained (MOE_FLAG_CHAIN: each launch may start under the
    # previous one), with the next layer's first shared-expert stages brought
    # into L2 during each launch's tail (moe_fused_decode_next), and both
    sh_c = B.make_shape(shape.T, shape.H, shape.I, shape.I_shared, shape.E, shape.K, args.flags | B.MOE_FLAG_CHAIN)

    def launch_c(i, s):
        rw, sw = weights[i % len(weights)]
        B.moe_fused_decode(L.x, L.topk_ids, L.topk_w, rw, sw, out, sh_c, ws, stream=s)

    def launch_n(i, s, sh_=sh):
        rw, sw = weights[i % len(weights)]
        nsw = weights[(i + 1) % len(weights)][1]
        B.moe_fused_decode_next(L.x, L.topk_ids, L.topk_w, rw, sw, nsw, out, sh_, ws, stream=s)

    def launch_nc(i, s):
        launch_n(i, s, sh_c)

    chain = None if args.no_chain else chain_ab(
        {"plain": launch_s, "chain": launch_c, "next": launch_n, "next_chain": launch_nc}, 4 * len(weights))
    assert B.moe_read_error(ws) == 0

    # the other workloads of the metric (T=8, T=64) and the routed T=1 layer,
    # unless --no-sweep
    del copies, weights
    torch.cuda.empty_cache()
    sweep = {}
    if not args.no_sweep:
        for name in WORKLOADS:
            if name == args.workload:
                continue
            sweep[name] = sweep_point(name, args, dev)
        for name in ROUTED:
            sweep[name] = routed_point(name, args, dev)
        for name, base in FP8_MID.items():
            sweep[name] = sweep_point(base, args, dev, B.MOE_FLAG_FP8_MID)
            sweep[name]["flags"] = "MOE_FLAG_FP8_MID"
    wide = wide_sweep(args, dev) if args.sweep_wide else {}
    clk2.__exit__()
    return dict(us_launch=us_launch_max, ms_per_step=ms_per_step, algo_bytes=algo_bytes,
                distinct=distinct, clocks=clk.summary(), err=err, e2e_us=e2e_us,
                h2d=xh.numel() * 2 + ih.numel() * 4 + wh.numel() * 4, d2h=oh.numel() * 2,
                sweep=sweep, wide=wide, graph_us=graph_us, T=shape.T, per_launch=per_launch, chain=chain,
                clocks_after=clk2.summary())


def graph_us_per_launch(launch, n_launch: int, reps: int = 5) -> float:
    """us per launch with `n_launch` launches captured in one CUDA graph and the
    graph replayed `reps` times (events on the capturing stream)."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        launch(0, s)  # warm (outside capture)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            for i in range(n_launch):
                launch(i, s)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        a.record(s)
        for _ in range(reps):
            g.replay()
        b.record(s)
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e3 / (reps * n_launch)


def capture_graph(launch, n_launch: int):
    """n_launch launches captured in one CUDA graph on a side stream."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        launch(0, s)  # warm (outside capture)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            for i in range(n_launch):
                launch(i, s)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    return g, s


def chain_ab(variants: dict, n_launch: int, rounds: int = 3, reps: int = 3) -> dict:
    """Layers back to back in several forms (name -> launch(i, stream)), all
    forms alternating within every round: eagerly (n_launch launches between
    two events) and as CUDA-graph replays. Medians over the rounds, us per
    launch: `<name>_us_per_launch` and `<name>_graph_us_per_launch`."""
    import torch
    st = torch.cuda.current_stream()

    def eager(f):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(HEAD_START_CYCLES)
        a.record(st)
        for i in range(n_launch):
            f(i, st)
        b.record(st)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / n_launch

    def replay(gs):
        g, s = gs
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            a.record(s)
            for _ in range(reps):
                g.replay()
            b.record(s)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / (reps * n_launch)

    for f in variants.values():
        for i in range(n_launch):
            f(i, st)
    torch.cuda.synchronize()
    graphs = {k: capture_graph(f, n_launch) for k, f in variants.items()}
    t = {}
    for _ in range(rounds):
        for k, f in variants.items():
            t.setdefault(f"{k}_us_per_launch", []).append(eager(f))
            t.setdefault(f"{k}_graph_us_per_launch", []).append(replay(graphs[k]))
    del graphs
    out = {k: round(statistics.median(v), 2) for k, v in t.items()}
    out["layers_back_to_back"] = n_launch
    out["rounds"] = rounds
    return out


def back_to_back_us(launch, n: int) -> float:
    """us per launch of n launches back to back on the current stream, between
    two events."""
    import torch
    st = torch.cuda.current_stream()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    torch.cuda._sleep(HEAD_START_CYCLES)
    a.record(st)
    for i in range(n):
        launch(i)
    b.record(st)
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e3 / n


def sweep_point(name, args, dev, extra_flags: int = 0):
    """us per launch for another workload (same protocol, fewer steps)."""
    import torch

    from moe_layer_decode_persistent_b300 import binding as B
    from moe_layer_decode_persistent_b300 import inputs
    wl = WORKLOADS[name]
    shape = inputs.dsv3(wl["T"], E=args.experts)
    L = inputs.make_layer(shape, wl["routing"], 0, dev, inputs.FMT_NVFP4, inputs.FMT_FP8_B128,
                          used_only=True)
    copies = [(L.routed, L.shared)] + [
        (inputs.ExpertSet(**{k: (v.clone() if isinstance(v, torch.Tensor) else v)
                             for k, v in L.routed.__dict__.items()}), L.shared)
        for _ in range(N_COPIES - 1)]
    weights = [(B.make_weights(r), B.make_weights(s)) for r, s in copies]
    sh = B.make_shape(shape.T, shape.H, shape.I, shape.I_shared, shape.E, shape.K, args.flags | extra_flags)
    ws = torch.empty(B.moe_workspace_bytes(sh), dtype=torch.uint8, device=dev)
    B.moe_workspace_init(ws)
    out = torch.empty(shape.T, shape.H, dtype=torch.bfloat16, device=dev)
    for i in range(3):
        B.moe_fused_decode(L.x, L.topk_ids, L.topk_w, *weights[i % N_COPIES], out, sh, ws)
    n = max(20, args.steps // 2)
    us = back_to_back_us(lambda i: B.moe_fused_decode(L.x, L.topk_ids, L.topk_w, *weights[i % N_COPIES], out,
                                                      sh, ws), n)
    assert B.moe_read_error(ws) == 0

    def launch_s(i, s):
        B.moe_fused_decode(L.x, L.topk_ids, L.topk_w, *weights[i % N_COPIES], out, sh, ws, stream=s)

    g_us = graph_us_per_launch(launch_s, 2 * N_COPIES)
    assert B.moe_read_error(ws) == 0
    b, distinct = algorithmic_bytes(L, L.topk_ids.cpu())
    peak, _ = measured_peaks()
    gbs = b / (us * 1e-6) / 1e9
    del L, copies, weights
    torch.cuda.empty_cache()
    return {"us_per_launch": round(us, 2), "graph_us_per_launch": round(g_us, 2), "hbm_gbs": round(gbs, 1),
            "frac": round(gbs / peak, 4), "frac_graph": round(b / (g_us * 1e-6) / 1e9 / peak, 4),
            "distinct_experts": distinct, "algo_bytes": b, "launches": n, "T": wl["T"],
            "routing": wl["routing"]}


def routed_point(name, args, dev):
    """us per launch of the layer with its router inside the launch
    (moe_fused_decode_routed): the same protocol as sweep_point. Every routed
    expert's weights are drawn, since the router picks them."""
    import torch

    from moe_layer_decode_persistent_b300 import binding as B
    from moe_layer_decode_persistent_b300 import inputs
    T = ROUTED[name]["T"]
    shape = inputs.dsv3(T, E=args.experts)
    L = inputs.make_layer(shape, "uniform", 0, dev, inputs.FMT_NVFP4, inputs.FMT_FP8_B128)
    g = torch.Generator(device=dev)
    g.manual_seed(1234)
    wr = (torch.randn(shape.E, shape.H, generator=g, device=dev) * (1.5 / shape.H ** 0.5)).to(torch.bfloat16)
    bias = (torch.randn(shape.E, generator=g, device=dev) * 0.05).to(torch.bfloat16)
    router = B.make_router(wr, bias, 2.5, True)
    copies = [(L.routed, L.shared)] + [
        (inputs.ExpertSet(**{k: (v.clone() if isinstance(v, torch.Tensor) else v)
                             for k, v in L.routed.__dict__.items()}), L.shared)
        for _ in range(N_COPIES - 1)]
    weights = [(B.make_weights(r), B.make_weights(s)) for r, s in copies]
    sh = B.make_shape(T, shape.H, shape.I, shape.I_shared, shape.E, shape.K, args.flags)
    ws = torch.empty(B.moe_workspace_bytes(sh), dtype=torch.uint8, device=dev)
    B.moe_workspace_init(ws)
    out = torch.empty(T, shape.H, dtype=torch.bfloat16, device=dev)
    ids = torch.empty(T, shape.K, dtype=torch.int32, device=dev)
    tw = torch.empty(T, shape.K, dtype=torch.float32, device=dev)

    def launch_s(i, s_=None):
        rw, sw = weights[i % N_COPIES]
        B.moe_fused_decode_routed(L.x, router, rw, sw, out, sh, ws, topk_ids=ids, topk_w=tw, stream=s_)

    for i in range(3):
        launch_s(i)
    n = max(20, args.steps // 2)
    us = back_to_back_us(launch_s, n)
    assert B.moe_read_error(ws) == 0
    g_us = graph_us_per_launch(launch_s, 2 * N_COPIES)
    assert B.moe_read_error(ws) == 0
    distinct = len(set(ids.cpu().reshape(-1).tolist()))
    b = (distinct * L.routed.nbytes_expert() + L.shared.nbytes_expert() + wr.numel() * 2 + bias.numel() * 2
         + 2 * T * shape.H * 2 + T * shape.K * 8)
    peak, _ = measured_peaks()
    gbs = b / (us * 1e-6) / 1e9
    del L, copies, weights
    torch.cuda.empty_cache()
    return {"us_per_launch": round(us, 2), "graph_us_per_launch": round(g_us, 2), "hbm_gbs": round(gbs, 1),
            "frac": round(gbs / peak, 4), "frac_graph": round(b / (g_us * 1e-6) / 1e9 / peak, 4),
            "distinct_experts": distinct, "algo_bytes": b, "launches": n, "T": T,
            "routing": "router inside the launch (sigmoid + bf16 correction bias, top-8, renormalised)"}


WIDE_T = [1, 2, 4, 8, 16, 32, 64, 128, 256]


def wide_sweep(args, dev, n_layers: int = 4):
    """Wide-expert layer (E=384 top-8, H=7168, I=2048, NVFP4 routed / FP8 shared,
    uniform routing): us per launch at each T, launches over n_layers distinct
    layers' resident weights run back to back."""
    import torch

    from moe_layer_decode_persistent_b300 import binding as B
    from moe_layer_decode_persistent_b300 import inputs
    E = 384
    base = inputs.dsv3(1, E=E)
    layers = []
    for l in range(n_layers):
        r = inputs.make_experts(inputs.FMT_NVFP4, E, base.H, base.I, ("L", l, 0), dev, tag="routed")
        s_ = inputs.make_experts(inputs.FMT_FP8_B128, 1, base.H, base.I_shared, ("L", l, 0), dev, tag="shared")
        layers.append((r, s_, B.make_weights(r), B.make_weights(s_)))
    peak, _ = measured_peaks()
    res = {}
    for T in WIDE_T:
        shape = inputs.dsv3(T, E=E)
        ids = inputs.ROUTINGS["uniform"](T, shape.K, E, 0).to(dev)
        w = inputs.router_weights(T, shape.K, 0).to(dev)
        x = inputs.activations(T, shape.H, 0, dev)
        sh = B.make_shape(T, shape.H, shape.I, shape.I_shared, E, shape.K, args.flags)
        ws = torch.empty(B.moe_workspace_bytes(sh), dtype=torch.uint8, device=dev)
        B.moe_workspace_init(ws)
        out = torch.empty(T, shape.H, dtype=torch.bfloat16, device=dev)

        def launch_s(i, s):
            _, _, rw, sw = layers[i % n_layers]
            B.moe_fused_decode(x, ids, w, rw, sw, out, sh, ws, stream=s)

        stream = torch.cuda.current_stream(dev)
        for i in range(2 * n_layers):
            launch_s(i, stream)
        n = 4 * n_layers
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        torch.cuda._sleep(HEAD_START_CYCLES)
        a.record(stream)
        for i in range(n):
            launch_s(i, stream)
        b.record(stream)
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / n
        g_us = graph_us_per_launch(launch_s, 2 * n_layers)
        sh_c = B.make_shape(T, shape.H, shape.I, shape.I_shared, E, shape.K, args.flags | B.MOE_FLAG_CHAIN)

        def launch_c(i, s, sh_c=sh_c, ws=ws, out=out, x=x, ids=ids, w=w):
            _, _, rw, sw = layers[i % n_layers]
            B.moe_fused_decode(x, ids, w, rw, sw, out, sh_c, ws, stream=s)

        def launch_n(i, s, sh_=sh, ws=ws, out=out, x=x, ids=ids, w=w):
            _, _, rw, sw = layers[i % n_layers]
            nsw = layers[(i + 1) % n_layers][3]
            B.moe_fused_decode_next(x, ids, w, rw, sw, nsw, out, sh_, ws, stream=s)

        chain = chain_ab({"plain": launch_s, "chain": launch_c, "next": launch_n,
                          "next_chain": lambda i, s_, sh_c=sh_c, f=launch_n: f(i, s_, sh_c)}, 2 * n_layers)
        assert B.moe_read_error(ws) == 0
        distinct = len(set(int(e) for e in ids.cpu().reshape(-1).tolist()))
        byt = distinct * layers[0][0].nbytes_expert() + layers[0][1].nbytes_expert() + 4 * T * shape.H + 8 * T * shape.K
        gbs = byt / (us * 1e-6) / 1e9
        res[str(T)] = {"us_per_launch": round(us, 2), "graph_us_per_launch": round(g_us, 2),
                       "hbm_gbs": round(gbs, 1), "frac": round(gbs / peak, 4), "distinct_experts": distinct,
                       "algo_bytes": byt, "chain_ab": chain}
        del ws, out
    del layers
    torch.cuda.empty_cache()
    return res


def oracle_launch(workload: str):
    """One whole launch of the workload for the CPU oracle: the batch's inputs
    and the experts it uses (drawn on the host with the GPU arm's recipe, the
    routed ones stored compactly), and a callable that runs the oracle on every
    row with the given thread count. Returns (run, expert uses per launch)."""
    import numpy as np

    import oracle
    from moe_layer_decode_persistent_b300 import inputs
    wl = WORKLOADS[workload]
    shape = inputs.dsv3(wl["T"])
    ids = inputs.ROUTINGS[wl["routing"]](shape.T, shape.K, shape.E, 0)
    used = sorted(set(int(e) for e in ids.reshape(-1).tolist()))
    remap = {e: i for i, e in enumerate(used)}
    ids_c = ids.clone()
    for t in range(shape.T):
        for p in range(shape.K):
            ids_c[t, p] = remap[int(ids[t, p])]
    routed = inputs.make_expert_subset(inputs.FMT_NVFP4, used, shape.H, shape.I, ("L", 0, 0), "cpu")
    shared = inputs.make_experts(inputs.FMT_FP8_B128, 1, shape.H, shape.I_shared, ("L", 0, 0), "cpu",
                                 tag="shared")

    def wset(es):
        return oracle.WeightSet(es.fmt, es.w13, es.w2, es.w13_scale, es.w2_scale, es.w13_gscale, es.w2_gscale)

    rw, sw = wset(routed), wset(shared)
    x = inputs.activations(shape.T, shape.H, 0)
    w = inputs.router_weights(shape.T, shape.K, 0)
    uses = shape.T * (shape.K + 1)

    def run(threads):
        out = oracle.moe_layer_uses(x, ids_c, w, rw, sw, shape.T, shape.H, shape.I, shape.I_shared,
                                    len(used), shape.K, threads=threads)
        assert np.isfinite(out).all()

    return run, uses


def oracle_threads(uses: int) -> int:
    return max(1, min(uses, os.cpu_count() or 1))


def run_reference(args):
    """The reference arm: the fp64 oracle, one whole launch of the workload
    per step, its expert evaluations spread over the host's cores."""
    import oracle
    oracle.build()
    run, uses = oracle_launch(args.workload)
    threads = oracle_threads(uses)
    for _ in range(args.warmup):
        run(threads)
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        run(threads)
        times.append(time.perf_counter() - t)
    return statistics.mean(times) * 1e6, threads, uses


def cpu_baseline(args):
    """The oracle as it stands, timed on this host: whole launches of the
    workload (all rows, every expert use), repeated for about 10 s."""
    import oracle
    oracle.build()
    run, uses = oracle_launch(args.workload)
    threads = oracle_threads(uses)
    run(threads)  # first touch of the weights
    t = time.perf_counter()
    n = 0
    while n < 1 or time.perf_counter() - t < 10.0:
        run(threads)
        n += 1
    us = (time.perf_counter() - t) / n * 1e6
    return {"value": round(us, 1), "unit": "us", "cores": threads, "host_cpus": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{n} whole {args.workload} launches (every row, {uses} expert evaluations "
                      f"each: dequant + SwiGLU + down in fp64, then the fixed-order sum), the "
                      f"evaluations of a launch spread over {threads} threads"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(WORKLOADS), default="dsv3_t1")
    ap.add_argument("--flags", type=int, default=0)
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the T=8 and T=64 workloads (timed by default, under `sweep`)")
    ap.add_argument("--sweep-wide", action="store_true",
                    help="also time the wide-expert layer (E=384) at T=1..256, 4 layers back to back")
    ap.add_argument("--no-chain", action="store_true",
                    help="skip the back-to-back forms (chained, next-layer prefetch) of the main workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer (end-to-end) timing")
    ap.add_argument("--experts", type=int, default=256,
                    help="routed experts E (profiling runs use fewer to bound device memory)")
    ap.add_argument("--copies", type=int, default=N_COPIES,
                    help="resident weight copies rotated per step")
    args = ap.parse_args()
    rank, world, local = dist_setup(args)
    T = WORKLOADS[args.workload]["T"]
    metric = "us per MoE-layer launch"
    config = {"workload": f"{args.workload}: DeepSeek-V3-shaped decode MoE layer, T={T}, H=7168, "
                          f"routed I=2048 NVFP4 E={args.experts} top-8, shared I=2048 FP8 128x128, "
                          f"{WORKLOADS[args.workload]['routing']} routing",
              "T": T, "l2": f"{args.copies} resident weight copies rotated per step (inputs larger than L2)"}

    if args.impl == "reference":
        if rank != 0:
            return
        us_launch, threads, uses = run_reference(args)
        line = {"impl": "reference", "metric": metric, "value": round(us_launch, 1), "unit": "us",
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(us_launch / 1e3, 3), "higher_is_better": False,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic (the same recipe, drawn on the host)", "config": config,
                "cpu_baseline": {"value": round(us_launch, 1), "unit": "us", "cores": threads,
                                 "host_cpus": os.cpu_count(), "kind": "oracle",
                                 "sample": f"every step one whole {args.workload} launch of the fp64 "
                                           f"oracle ({uses} expert evaluations over {threads} "
                                           f"threads, then the fixed-order sum of every row)"},
                "e2e": {"value": round(us_launch, 1), "unit": "us", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    r = run_ours(args, rank, world, local)
    if rank != 0:
        return
    peak, peak_kind = measured_peaks()
    gbs = r["algo_bytes"] / (r["us_launch"] * 1e-6) / 1e9
    kname = "fused_fma_kernel" if (args.flags & 2) else "fused_tc_kernel"
    trec = traffic_record(kname)
    line = {
        "metric": metric, "value": round(r["us_launch"], 2), "unit": "us", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(r["ms_per_step"], 4),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "fp32",
        "data": "synthetic (seeded N(0,0.02) weights encoded to NVFP4/FP8, bf16 N(0,1) x)",
        "config": config,
        "hbm_gbs": round(gbs, 1), "distinct_experts": r["distinct"], "algo_bytes": r["algo_bytes"],
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(gbs / peak, 4), "peak_kind": peak_kind,
                     "traffic": (trec or {}).get("dram_bytes_per_launch"),
                     "kernel": kname},
        "e2e": None if r["e2e_us"] is None else
        {"value": round(r["e2e_us"], 2), "unit": "us", "h2d_bytes_per_step": r["h2d"],
         "d2h_bytes_per_step": r["d2h"]},
        "gpu_launches": args.steps, "clocks": r["clocks"], "device_error_word": r["err"],
        "graph_us_per_launch": None if r["graph_us"] is None else round(r["graph_us"], 2),
        "single_launch_us": {"median": round(statistics.median(r["per_launch"]), 2),
                             "min": round(min(r["per_launch"]), 2), "max": round(max(r["per_launch"]), 2),
                             "how": "an event pair around each launch, after the timed region"},
    }
    if r.get("clocks_after"):
        line["clocks_after_timed_region"] = r["clocks_after"]  # graph, chained and sweep timings
    if r["chain"]:
        line["chain"] = r["chain"]
    if r["sweep"]:
        line["sweep"] = r["sweep"]
    if r["wide"]:
        line["wide_sweep"] = r["wide"]
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
