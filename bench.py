#!/usr/bin/env python
"""Benchmark of the int4 routed-expert MoE block on GB300.

Metric: MoE-layer tokens/s (token passes through one MoE layer per second)
and the achieved HBM bandwidth, unique expert bytes touched / time, against
the measured copy bandwidth.  The default workload is the 80B-class decode
stack, the largest decode configuration that fits one GPU: E=512, k=10,
hidden 2048, inter 512, group 64, 48 layers, one token per step, each layer
with its own weights (44 GB resident).

One step = one token through all the stacked layers, replayed from a CUDA
graph of the library's launch sequence; the inputs of 16 distinct steps
rotate, and every step touches far more distinct expert bytes than the L2
holds.  Rank 0 prints one JSON line.

  python bench.py [--steps K] [--warmup W] [--workload 2]     # our CUDA path
  python bench.py --impl reference                            # the CPU oracle
Under torchrun each rank runs an independent replica (no collective on the
data path); the time is the max over ranks.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE-layer tokens/s and achieved HBM GB/s vs peak (int4 experts, 1 GB300)"
UNIT = "layer-tokens/s"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", type=int, default=2,
                   help="synthetic workload (synth.WORKLOADS); 2 = 80B-class decode stack")
    p.add_argument("--layers", type=int, default=None, help="override the stack depth")
    p.add_argument("--distinct", type=int, default=16, help="distinct step inputs")
    p.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle timing")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--path", type=int, default=0, help="kernel path (0 auto)")
    p.add_argument("--mode", choices=["auto", "stack", "layers", "gdn"], default="auto",
                   help="one-token workloads: 'stack' chains the layers (RMSNorm + residual) "
                        "in one persistent launch per token; 'layers' runs independent "
                        "layers, one moe_forward each (auto: stack)")
    p.add_argument("--bits", type=int, choices=[4, 8], default=4,
                   help="expert code width (8: int8 experts, the general path, --mode layers)")
    p.add_argument("--gdn-batch", type=int, default=64,
                   help="--mode gdn: independent sequences per launch")
    p.add_argument("--gdn-tokens", type=int, default=1,
                   help="--mode gdn: tokens per sequence per launch (1 = decode)")
    p.add_argument("--gdn-layers", type=int, default=36,
                   help="--mode gdn: Gated DeltaNet layers per step (own state each)")
    p.add_argument("--pool-slots", type=int, default=0,
                   help="bounded slot pool of this many resident experts per layer (the rest "
                        "in pinned host memory, LFU + recency eviction); implies --mode layers")
    p.add_argument("--phases", action="store_true",
                   help="one-token stacks: build the instrumented library (per-phase SM cycle "
                        "stamps) and print each phase's duration instead of the bench line")
    p.add_argument("--profile", action="store_true",
                   help="short run for profilers: no clock-warming loop, no end-to-end or "
                        "stage timing, no CPU baseline")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(ms, world, device):
    """The slowest replica's time: the whole job ends when the last rank does."""
    if world == 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(t_max_ms, world, tokens, layers, steps):
    """Layer-tokens per second of the whole job: every replica runs the same steps."""
    return world * tokens * layers * steps / (t_max_ms / 1e3)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            m = json.load(f)
        return {"hbm_gbs": float(m["hbm_gbs"]), "bf16_tflops": float(m["bf16_tflops"]),
                "bf16_tflops_sustained": float(m.get("bf16_tflops_sustained", m["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# DRAM bytes per launch of the dominant kernels, from ncu captures
# (profiles/traffic.json), with the hash of the sources they were taken on:
# reported only while those sources are unchanged.
TRAFFIC_SOURCES = {
    "decode_kernel": ["decode.cu", "gemv_mma.cuh", "routing_common.cuh", "device_util.cuh",
                      "sm100_ptx.cuh", "moe_internal.cuh"],
    "fused_decode_kernel": ["fused_decode.cu", "routing_common.cuh", "device_util.cuh",
                            "sm100_ptx.cuh", "moe_internal.cuh"],
    "gdn_recurrence_kernel": ["gdn.cu", "sm100_ptx.cuh"],
    "grouped_gemm_kernel<gate/up>": ["prefill.cu", "device_util.cuh", "sm100_ptx.cuh",
                                     "moe_internal.cuh"],
}


def sources_sha256(kernel):
    import hashlib
    h = hashlib.sha256()
    for f in TRAFFIC_SOURCES[kernel]:
        with open(os.path.join(ROOT, "int4_routed_expert_decode_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic(kernel, workload):
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)[kernel]
    except Exception:
        return None
    if t.get("workload") != workload or t.get("sources_sha256") != sources_sha256(kernel):
        return None
    return t.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [s.strip() for s in line.split(",")]
                    if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                        rows.append(parts)
            os.unlink(self.path)
        except Exception:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())
                if any(r[3].replace(".", "").isdigit() for r in rows) else None}


# --------------------------------------------------------------------- oracle timing
def oracle_units(wl, budget_s, layers, stacked, threads=0):
    """Time the C++ CPU oracle (OpenMP; `threads` 0 = all cores) on (layer,
    token) passes of the workload for about budget_s seconds.  A stack pass
    includes the RMSNorm and the residual add.  Returns (passes/s, passes,
    seconds, sample text)."""
    from oracle import cpp as C
    n_layers = min(layers, 2)
    Ws = [synth.layer_weights(0, wl.wid, l, wl.shape, zipf_s=wl.zipf_s) for l in range(n_layers)]
    norms = stack_norm_weights(wl, n_layers)
    tok = 1 if wl.T == 1 else min(wl.T, 8)
    x_state = synth.tokens(0, wl.wid, 0, 0, 1, wl.H)[0]
    done = 0
    C.load()  # compile outside the timed region
    t0 = time.perf_counter()
    step = 0
    while True:
        l = step % n_layers
        if stacked:
            r = C.moe_stack(x_state, [Ws[l]], [norms[l]], wl.k, wl.G, STACK_EPS, threads=threads)
            x_state = r["x"][1]
        else:
            x = synth.tokens(0, wl.wid, l, step // n_layers, wl.T, wl.H)
            C.moe_block(x, Ws[l], wl.k, wl.G, tokens=list(range(tok)), threads=threads)
        done += tok
        step += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    sample = (f"{done} (layer, token) passes of the C++ oracle over layers 0..{n_layers - 1}, "
              f"{tok} token(s) per pass" + ("" if wl.T == 1 else f" of a {wl.T}-token batch") +
              (" (RMSNorm and residual included)" if stacked else ""))
    return done / dt, done, dt, sample


def cpu_baseline(wl, budget_s, L, stacked):
    """The oracle on all host cores, and on one core for a single-thread figure."""
    v, n, dt, sample = oracle_units(wl, budget_s * 0.7, L, stacked, threads=0)
    v1, n1, dt1, _ = oracle_units(wl, budget_s * 0.3, L, stacked, threads=1)
    return {"value": v, "unit": UNIT, "cores": cores_used(), "kind": "oracle",
            "sample": sample + f", {dt:.1f} s on {cores_used()} threads",
            "single_thread": {"value": v1, "unit": UNIT, "cores": 1,
                              "sample": f"{n1} passes, {dt1:.1f} s"}}


def cores_used():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# --------------------------------------------------------------------- reference arm
def run_reference(args, wl):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from oracle import cpp as C
    L = args.layers or wl.layers
    n_layers = min(L, 2)
    Ws = [synth.layer_weights(0, wl.wid, l, wl.shape, zipf_s=wl.zipf_s) for l in range(n_layers)]
    tok = 1 if wl.T == 1 else min(wl.T, 8)
    stacked = stack_mode(args, wl)
    norms = stack_norm_weights(wl, n_layers)
    state = {"x": synth.tokens(0, wl.wid, 0, 0, 1, wl.H)[0]}
    C.load()  # compiled before timing

    def step(i):
        l = i % n_layers
        if stacked:  # one layer of the residual stack: RMSNorm, block, residual add
            r = C.moe_stack(state["x"], [Ws[l]], [norms[l]], wl.k, wl.G, STACK_EPS)
            state["x"] = r["x"][1]
            return
        x = synth.tokens(0, wl.wid, l, i // n_layers, wl.T, wl.H)
        C.moe_block(x, Ws[l], wl.k, wl.G, tokens=list(range(tok)))

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = args.steps * tok / dt
    sample = (f"each step: {tok} token(s) through one MoE layer (layers 0..{n_layers - 1} "
              "alternate)" + (", with the stack's RMSNorm and residual add" if stacked else ""))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": config_of(wl, L, stacked),
        "note": "C++ CPU oracle (float64, OpenMP on all host cores), a bounded sample of the "
                "workload per step",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores_used(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def stack_mode(args, wl):
    return wl.T == 1 and args.mode in ("auto", "stack") and not args.pool_slots and args.bits == 4


STACK_EPS = 1e-6


def stack_norm_weights(wl, L):
    """Seeded RMSNorm weights of the stack, bf16 bits ~ N(1, 0.1^2) (synthetic)."""
    return [synth.norm_weights(0, wl.wid, l, wl.H) for l in range(L)]


def config_of(wl, L, stacked, bits=4):
    """The workload's description; both arms print the same dict."""
    return {"workload": wl.name + ("-int8" if bits == 8 else ""), "E": wl.E, "k": wl.k,
            "hidden": wl.H, "inter": wl.I,
            "shared_inter": wl.Is, "group": wl.G, "tokens_per_step": wl.T, "layers": L,
            "zipf_s": wl.zipf_s,
            "chaining": "layer l+1 consumes RMSNorm(x_l + y_l) (residual stack)" if stacked
                        else "independent layers, each with its own seeded input",
            "weights": f"int{bits} affine (bf16 scale+bias per group), seeded synthetic",
            "parallelism": "replicas",
            "l2": "inputs larger than L2: every step streams distinct expert weights "
                  "far beyond the 129 MB L2; distinct step inputs rotate"}


# --------------------------------------------------------------------- our arm
STAGES = ("router", "topk", "permute", "gateup", "down", "combine")


def stage_times(moe, torch, ctx, enqueue, inputs, stream, k):
    """Mean device time of each stage of the first layer's moe_forward over k
    eager steps, from the library's stage events (recorded on the launching
    stream).  Stages a path does not have are absent."""
    sets = []
    with torch.cuda.stream(stream):
        for i in range(k):
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(moe.MOE_MARK_COUNT)]
            for e in evs:
                e.record(stream)  # creates the event; a later record by the library moves it
            sets.append(evs)
        stream.synchronize()
        for i in range(k):
            moe.moe_set_stage_events(ctx, sets[i])
            enqueue(inputs[i % len(inputs)])
        moe.moe_set_stage_events(ctx, [])
        stream.synchronize()
    acc = {}
    for evs in sets:
        marks = [0.0] + [evs[0].elapsed_time(evs[m]) for m in range(1, moe.MOE_MARK_COUNT)]
        seen = [m for m in range(moe.MOE_MARK_COUNT) if m == 0 or marks[m] >= 0.0]
        for a, b in zip(seen, seen[1:]):
            name = STAGES[a] if b == a + 1 else "+".join(STAGES[a:b])
            acc.setdefault(name, []).append((marks[b] - marks[a]) * 1e3)
        acc.setdefault("total", []).append(marks[moe.MOE_MARK_END] * 1e3)
    return {n: float(np.mean(v)) for n, v in acc.items()}


def run_ours(args, wl):
    import torch

    import int4_routed_expert_decode_gb300 as moe
    from int4_routed_expert_decode_gb300 import build as moe_build

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    moe_build.build()
    L = args.layers or wl.layers
    T, H = wl.T, wl.H
    S = max(1, min(args.distinct, args.steps + args.warmup))
    layers = []
    weights_of = synth.layer_weights_int8 if args.bits == 8 else synth.layer_weights
    for l in range(L):
        W = weights_of(0, wl.wid, l, wl.shape, zipf_s=wl.zipf_s)
        layer = moe.MoELayer(wl.E, wl.k, H, wl.I, wl.Is, wl.G, weights=W, max_T=T,
                             bits=args.bits)
        if args.path:
            moe.moe_set_path(layer.ctx, args.path)
        if args.pool_slots:
            moe.moe_pool_enable(layer.ctx, args.pool_slots)
        layers.append(layer)
        del W
    x_all = torch.empty((S, L, T, H), dtype=torch.bfloat16, device="cuda")
    for s in range(S):
        for l in range(L):
            xs = synth.tokens(0, wl.wid, l, s, T, H)
            x_all[s, l].copy_(torch.from_numpy(xs.view(np.int16)).view(torch.bfloat16))
    y = torch.empty((L, T, H), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((L, T, wl.k), dtype=torch.int32, device="cuda")
    wts = torch.empty((L, T, wl.k), dtype=torch.float32, device="cuda")
    x_in = torch.empty((L, T, H), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.Stream()

    def enqueue(xsrc):
        for l in range(L):
            moe.moe_forward(layers[l].ctx, xsrc[l], T, None, y[l], idx[l], wts[l],
                            stream=stream.cuda_stream)

    # eager pass per distinct input: statuses, unique experts, launch count
    # (int8 codes take twice the int4 code bytes)
    e_bytes = wl.expert_bytes + (3 * wl.I * wl.H // 2 if args.bits == 8 else 0)
    s_bytes = wl.shared_bytes + (3 * wl.Is * wl.H // 2 if args.bits == 8 else 0)
    uniq_bytes = []
    ys0 = None
    with torch.cuda.stream(stream):
        for s in range(S):
            enqueue(x_all[s])
            stream.synchronize()
            if s == 0:
                ys0 = y.clone()
            ids = idx.cpu().numpy()
            uniq_bytes.append(sum(len(set(ids[l].ravel().tolist())) * e_bytes + s_bytes
                                  for l in range(L)))
    for l in range(L):
        st = layers[l].status(stream.cuda_stream)
        if st != moe.MOE_OK:
            raise RuntimeError(f"layer {l}: {moe.moe_status_string(st)}")
    launches_per_layer = moe.moe_last_launch_count(layers[-1].ctx)
    unique_per_step = float(np.mean(uniq_bytes))

    graphs = []
    for s in range(S):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            enqueue(x_all[s])
        graphs.append(g)
    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_e2e, stream=stream):
        enqueue(x_in)

    clocks = ClockSampler(local).start()
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            graphs[i % S].replay()
        stream.synchronize()
        # keep the GPU loaded ~1 s so that clock samples exist before timing
        t_load = time.perf_counter()
        i = 0
        while not args.profile and time.perf_counter() - t_load < 1.0:
            graphs[i % S].replay()
            i += 1
            if i % 64 == 0:
                stream.synchronize()
        stream.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        pool0 = [moe.moe_pool_stats(l.ctx) for l in layers] if args.pool_slots else None
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for i in range(args.steps):
            graphs[(args.warmup + i) % S].replay()
        ev1.record(stream)
        ev1.synchronize()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        ms = ev0.elapsed_time(ev1)
        pool = None
        if args.pool_slots:
            pool1 = [moe.moe_pool_stats(l.ctx) for l in layers]
            hits = sum(b["hits"] - a["hits"] for a, b in zip(pool0, pool1))
            misses = sum(b["misses"] - a["misses"] for a, b in zip(pool0, pool1))
            pool = {"slots_per_layer": args.pool_slots, "experts_per_layer": wl.E,
                    "hit_rate": hits / max(1, hits + misses), "hits": hits, "misses": misses,
                    "fills_from_pinned_host_per_step": misses / args.steps,
                    "overflows": sum(b["overflows"] - a["overflows"]
                                     for a, b in zip(pool0, pool1)),
                    "distinct_step_inputs": S}
    clk = clocks.stop()
    # per-stage device times of layer 0 (eager, same stream, after the timed region)
    stages = {} if args.profile else stage_times(
        moe, torch, layers[0].ctx, enqueue, [x_all[s] for s in range(S)], stream,
        k=max(3, min(args.steps, 20)))
    t_max = max_over_ranks(ms, world, "cuda")
    value = job_throughput(t_max, world, T, L, args.steps)
    ms_step = t_max / args.steps
    us_layer = ms_step * 1e3 / L
    hbm = unique_per_step / (ms_step / 1e3) / 1e9
    pk = peaks()

    # e2e through the C ABI with host buffers: H2D x, graph, D2H y every step
    x_host = torch.empty((L, T, H), dtype=torch.bfloat16, pin_memory=True)
    x_host.copy_(x_all[0].cpu())
    y_host = torch.empty((L, T, H), dtype=torch.bfloat16, pin_memory=True)
    k_e2e = 1 if args.profile else max(1, min(args.steps, 200))
    with torch.cuda.stream(stream):
        for _ in range(3):
            x_in.copy_(x_host, non_blocking=True)
            g_e2e.replay()
            y_host.copy_(y, non_blocking=True)
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(k_e2e):
            x_in.copy_(x_host, non_blocking=True)
            g_e2e.replay()
            y_host.copy_(y, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        ms_e2e = e0.elapsed_time(e1) / k_e2e
    e2e_value = world * T * L / (ms_e2e / 1e3)

    # C++ oracle on the host cores (rank 0, N = 1), and a parity spot check of
    # layer 0's first eager step against the numpy oracle
    cpu = None
    parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.profile:
        from oracle import moe_oracle as O
        W0 = weights_of(0, wl.wid, 0, wl.shape, zipf_s=wl.zipf_s)
        if args.bits == 4:
            cpu = cpu_baseline(wl, args.cpu_budget, L, False)
        else:  # the int8 block's oracle is the numpy one, one core
            n, t0 = 0, time.perf_counter()
            while time.perf_counter() - t0 < min(args.cpu_budget, 10.0):
                O.moe_block(synth.tokens(0, wl.wid, 0, n, 1, H), W0, wl.k, wl.G)
                n += 1
            cpu = {"value": n / (time.perf_counter() - t0), "unit": UNIT, "cores": 1,
                   "kind": "oracle", "sample": f"{n} layer-tokens of layer 0 through the numpy "
                                               "float64 oracle (int8 experts)"}
        rows = list(range(min(T, 4)))
        r = O.moe_block(synth.tokens(0, wl.wid, 0, 0, T, H), W0, wl.k, wl.G, tokens=rows)
        yg = ys0[0, rows].float().cpu().numpy().astype(np.float64)
        parity = {"checked": f"layer 0, rows {rows}",
                  "max_rel_err": float(np.abs(yg - r["y"]).max() / np.abs(r["y"]).max())}

    P = T * wl.k
    flops = {"gateup": 2.0 * H * (2 * wl.I * P + 2 * wl.Is * T),
             "down": 2.0 * H * (wl.I * P + wl.Is * T), "router": 2.0 * H * wl.E * T}
    flops_layer = sum(flops.values())
    grouped = args.bits == 4 and (args.path == 3 or (args.path == 0 and T > 1))  # tcgen05 GEMMs
    # up to 64 tokens a layer streams each selected expert once for few tokens: HBM bound;
    # thousands of tokens make the grouped GEMMs tensor-core bound
    if grouped and T > 64 and "gateup" in stages:
        # many tokens: the grouped GEMMs are tensor-core bound; the gate/up GEMM dominates
        t_gu = stages["gateup"] * 1e-6
        achieved = flops["gateup"] / t_gu / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"],
                    "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"],
                    "traffic": measured_traffic("grouped_gemm_kernel<gate/up>", wl.name),
                    "kernel": "grouped_gemm_kernel<gate/up> (tcgen05 bf16, fp32 TMEM), "
                              f"{flops['gateup'] / 1e9:.1f} GFLOP algorithmic per launch, "
                              f"{stages['gateup']:.1f} us per launch",
                    "peak_source": pk["source"] + " burst bf16 (cuBLAS)"}
    else:
        algo_bytes_layer = unique_per_step / L + wl.router_bytes + 2 * T * H * 2
        achieved = algo_bytes_layer / (us_layer * 1e-6) / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                    "frac": achieved / pk["hbm_gbs"],
                    "traffic": measured_traffic("fused_decode_kernel", wl.name)
                    if launches_per_layer == 1 else None,
                    "kernel": f"one layer of moe_forward ({launches_per_layer} launches), "
                              f"{algo_bytes_layer / 1e6:.2f} MB algorithmic per layer",
                    "peak_source": pk["source"]}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if grouped else "fp32", "data": "synthetic",
        "config": config_of(wl, L, False, args.bits),
        "note": f"each step touches {unique_per_step / 1e6:.0f} MB of distinct expert weights; "
                f"{S} distinct step inputs rotate",
        "us_per_layer": us_layer, "stack_tokens_per_s": world * T / (ms_step / 1e3),
        "hbm_gbs_unique_expert_bytes": hbm, "hbm_frac": hbm / pk["hbm_gbs"],
        "tflops_layer": flops_layer / (us_layer * 1e-6) / 1e12,
        "stages_us_layer0": stages,
        "roofline": roofline, "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": L * T * H * 2,
                "d2h_bytes_per_step": L * T * H * 2},
        "clocks": clk, "gpu_launches": args.steps * L * launches_per_layer,
        "parity_spot_check": parity,
    }
    if pool is not None:
        line["pool"] = pool
    if rank == 0:
        print(json.dumps(line), flush=True)
    for layer in layers:
        layer.close()
    if world > 1:
        torch.distributed.destroy_process_group()


def run_ours_stack(args, wl):
    """One token per step through the whole residual stack: one persistent
    launch (moe_stack_forward) per step."""
    import torch

    import int4_routed_expert_decode_gb300 as moe
    from int4_routed_expert_decode_gb300 import build as moe_build

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    moe_build.build()
    L = args.layers or wl.layers
    H = wl.H
    S = max(1, min(args.distinct, args.steps + args.warmup))
    layers = []
    for l in range(L):
        W = synth.layer_weights(0, wl.wid, l, wl.shape, zipf_s=wl.zipf_s)
        layers.append(moe.MoELayer(wl.E, wl.k, H, wl.I, wl.Is, wl.G, weights=W, max_T=1))
        del W
    norms = [torch.from_numpy(g.view(np.int16)).cuda().view(torch.bfloat16)
             for g in stack_norm_weights(wl, L)]
    stack = moe.MoEStack(layers, norms, STACK_EPS)
    x_all = torch.empty((S, H), dtype=torch.bfloat16, device="cuda")
    for s in range(S):
        x_all[s].copy_(torch.from_numpy(synth.tokens(0, wl.wid, 0, s, 1, H)[0].view(np.int16))
                       .view(torch.bfloat16))
    x_out = torch.empty((H,), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((L, H), dtype=torch.bfloat16, device="cuda")
    xn = torch.empty((L, H), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((L, wl.k), dtype=torch.int32, device="cuda")
    wts = torch.empty((L, wl.k), dtype=torch.float32, device="cuda")
    x_in = torch.empty((H,), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.Stream()

    def enqueue(xsrc):
        moe.moe_stack_forward(stack.stack, xsrc, None, x_out, y, xn, idx, wts,
                              stream=stream.cuda_stream)

    uniq_bytes = []
    first = None
    with torch.cuda.stream(stream):
        for s in range(S):
            enqueue(x_all[s])
            stream.synchronize()
            if s == 0:
                first = (y.clone(), xn.clone(), idx.clone())
            ids = idx.cpu().numpy()
            uniq_bytes.append(sum(len(set(ids[l].tolist())) * wl.expert_bytes + wl.shared_bytes
                                  for l in range(L)))
    st = stack.status(stream.cuda_stream)
    if st != moe.MOE_OK:
        raise RuntimeError(f"stack: {moe.moe_status_string(st)}")
    unique_per_step = float(np.mean(uniq_bytes))

    clocks = ClockSampler(local).start()
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            enqueue(x_all[i % S])
        stream.synchronize()
        t_load = time.perf_counter()
        i = 0
        while not args.profile and time.perf_counter() - t_load < 1.0:
            enqueue(x_all[i % S])
            i += 1
            if i % 16 == 0:
                stream.synchronize()
        stream.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for i in range(args.steps):
            enqueue(x_all[(args.warmup + i) % S])
        ev1.record(stream)
        ev1.synchronize()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        ms = ev0.elapsed_time(ev1)
    clk = clocks.stop()
    st = stack.status(stream.cuda_stream)
    if st != moe.MOE_OK:
        raise RuntimeError(f"stack (timed): {moe.moe_status_string(st)}")
    t_max = max_over_ranks(ms, world, "cuda")
    value = job_throughput(t_max, world, 1, L, args.steps)
    ms_step = t_max / args.steps
    us_layer = ms_step * 1e3 / L
    hbm = unique_per_step / (ms_step / 1e3) / 1e9
    pk = peaks()

    # e2e through the C ABI with host buffers: H2D x, the launch, D2H x_out every step
    x_host = torch.empty((H,), dtype=torch.bfloat16, pin_memory=True)
    x_host.copy_(x_all[0].cpu())
    out_host = torch.empty((H,), dtype=torch.bfloat16, pin_memory=True)
    k_e2e = 1 if args.profile else max(1, min(args.steps, 200))
    with torch.cuda.stream(stream):
        for _ in range(3):
            x_in.copy_(x_host, non_blocking=True)
            enqueue(x_in)
            out_host.copy_(x_out, non_blocking=True)
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(k_e2e):
            x_in.copy_(x_host, non_blocking=True)
            enqueue(x_in)
            out_host.copy_(x_out, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        ms_e2e = e0.elapsed_time(e1) / k_e2e
    e2e_value = world * L / (ms_e2e / 1e3)

    cpu = None
    parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.profile:
        cpu = cpu_baseline(wl, args.cpu_budget, L, True)
        # layers 0 and L-1 of the first step against the oracle on the GPU's block input
        from oracle import moe_oracle as O
        y0, xn0, idx0 = first
        errs, idx_ok = [], True
        for l in sorted({0, L - 1}):
            W = synth.layer_weights(0, wl.wid, l, wl.shape, zipf_s=wl.zipf_s)
            nb = xn0[l].view(torch.int16).cpu().numpy().view(np.uint16)
            r = O.moe_block(nb[None, :], W, wl.k, wl.G)
            yg = y0[l].float().cpu().numpy().astype(np.float64)
            errs.append(float(np.abs(yg - r["y"][0]).max() / np.abs(r["y"][0]).max()))
            idx_ok = idx_ok and idx0[l].cpu().numpy().tolist() == r["topk_idx"][0].tolist()
        parity = {"checked_layers": sorted({0, L - 1}), "max_rel_err": max(errs),
                  "topk_idx_equal": idx_ok}

    P = wl.k
    flops_layer = 2.0 * H * (3 * wl.I * P + 3 * wl.Is + wl.E)
    algo_bytes_layer = unique_per_step / L + wl.router_bytes + 2 * H * 2
    achieved = algo_bytes_layer / (us_layer * 1e-6) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"],
                "traffic": measured_traffic("decode_kernel", wl.name),
                "kernel": f"decode_kernel, {L} layers per launch, "
                          f"{algo_bytes_layer / 1e6:.2f} MB algorithmic per layer "
                          f"({us_layer:.2f} us per layer)",
                "peak_source": pk["source"]}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp32", "data": "synthetic",
        "config": config_of(wl, L, True),
        "note": f"each step touches {unique_per_step / 1e6:.0f} MB of distinct expert weights; "
                f"{S} distinct step inputs rotate; one launch per step for all {L} layers",
        "us_per_layer": us_layer, "stack_tokens_per_s": world / (ms_step / 1e3),
        "hbm_gbs_unique_expert_bytes": hbm, "hbm_frac": hbm / pk["hbm_gbs"],
        "tflops_layer": flops_layer / (us_layer * 1e-6) / 1e12,
        "roofline": roofline, "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": H * 2,
                "d2h_bytes_per_step": H * 2},
        "clocks": clk, "gpu_launches": args.steps,
        "parity_spot_check": parity,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    stack.close()
    for layer in layers:
        layer.close()
    if world > 1:
        torch.distributed.destroy_process_group()


GDN_SHAPE = synth.GdnShape(Hk=16, Hv=32, dk=128, dv=128)


def gdn_oracle_rate(budget_s, Lg):
    """The float64 oracle on whole sequence-layers of the decode workload
    (one token each) for about budget_s seconds: sequence-layers/s."""
    from oracle import gdn_oracle as G
    done, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        q, k, v, a, b, S0 = synth.gdn_inputs(0, done % Lg, 1, 1, GDN_SHAPE, step=done)
        G.gdn_recurrence(q, k, v, a, b, S0)
        done += 1
    return done / (time.perf_counter() - t0), done


def run_gdn(args):
    """Gated DeltaNet decode: every step runs `gdn_layers` launches, one per
    layer, each advancing B sequences by T tokens with its own state."""
    import torch

    import int4_routed_expert_decode_gb300 as moe
    from int4_routed_expert_decode_gb300 import build as moe_build

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    moe_build.build()
    s, B, T, Lg = GDN_SHAPE, args.gdn_batch, args.gdn_tokens, args.gdn_layers

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16 if a.dtype == np.uint16
                                                            else a.dtype)).cuda()

    # Per layer its own state buffer (layers past the first few start from a
    # device copy of an earlier layer's seeded state); the token inputs of a
    # few distinct seeded draws rotate over layers and steps.
    S = max(1, min(args.distinct, 4, Lg))
    states, ins = [], []
    for l in range(S):
        q, k, v, a, b, S0 = synth.gdn_inputs(0, l, B, T, s)
        states.append(dev(S0))
        ins.append(tuple(dev(x) for x in (q, k, v, a, b)))
    for l in range(S, Lg):
        states.append(states[l % S].clone())
    out = torch.empty((B, T, s.Hv, s.dv), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()

    def enqueue(step, inputs=None):
        for l in range(Lg):
            q, k, v, a, b = inputs or ins[(step + l) % len(ins)]
            moe.moe_gdn_recurrence(q, k, v, a, b, states[l], out, B, T, s.Hk, s.Hv, s.dk, s.dv,
                                   stream=stream.cuda_stream)

    # parity spot check of sequence 0 and B-1 of layer 0, first step, against the oracle
    parity = None
    if rank == 0 and not args.profile:
        from oracle import gdn_oracle as G
        q, k, v, a, b, S0 = synth.gdn_inputs(0, 0, B, T, s)
        with torch.cuda.stream(stream):
            st0 = states[0].clone()
            o0 = torch.empty_like(out)
            qd, kd, vd, ad, bd = ins[0]
            moe.moe_gdn_recurrence(qd, kd, vd, ad, bd, st0, o0, B, T, s.Hk, s.Hv, s.dk, s.dv,
                                   stream=stream.cuda_stream)
            stream.synchronize()
        errs = []
        for i in sorted({0, B - 1}):
            ro, rS = G.gdn_recurrence(q[i:i + 1], k[i:i + 1], v[i:i + 1], a[i:i + 1], b[i:i + 1],
                                      S0[i:i + 1])
            scale = max(1.0, float(np.abs(rS).max()))
            errs.append(max(float(np.abs(o0[i].cpu().numpy() - ro[0]).max()),
                            float(np.abs(st0[i].cpu().numpy() - rS[0]).max())) / scale)
        parity = {"checked_sequences": sorted({0, B - 1}), "max_rel_err": max(errs)}

    clocks = ClockSampler(local).start()
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            enqueue(i)
        stream.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for i in range(args.steps):
            enqueue(args.warmup + i)
        ev1.record(stream)
        ev1.synchronize()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        ms = ev0.elapsed_time(ev1)
    clk = clocks.stop()
    t_max = max_over_ranks(ms, world, "cuda")
    ms_step = t_max / args.steps
    units = world * B * Lg * args.steps  # sequence-layers advanced by T tokens
    value = units / (t_max / 1e3)
    us_launch = ms_step * 1e3 / Lg
    state_bytes = B * s.Hv * s.dv * s.dk * 4
    in_bytes = B * T * (2 * s.Hk * s.dk * 2 + s.Hv * s.dv * 2 + 2 * s.Hv * 4)
    out_bytes = B * T * s.Hv * s.dv * 4
    algo = 2 * state_bytes + in_bytes + out_bytes
    pk = peaks()
    achieved = algo / (us_launch * 1e-6) / 1e9

    # e2e: host inputs in and the outputs back, every launch, pinned buffers
    hin = [x.cpu().pin_memory() for x in ins[0]]
    din = [torch.empty_like(x) for x in ins[0]]
    hout = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    k_e2e = 1 if args.profile else max(1, min(args.steps, 20))
    with torch.cuda.stream(stream):
        def e2e_step():
            for l in range(Lg):
                for d, h in zip(din, hin):
                    d.copy_(h, non_blocking=True)
                q, k, v, a, b = din
                moe.moe_gdn_recurrence(q, k, v, a, b, states[l], out, B, T, s.Hk, s.Hv, s.dk,
                                       s.dv, stream=stream.cuda_stream)
                hout.copy_(out, non_blocking=True)
        for _ in range(2):
            e2e_step()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(k_e2e):
            e2e_step()
        e1.record(stream)
        e1.synchronize()
        ms_e2e = e0.elapsed_time(e1) / k_e2e
    e2e = {"value": world * B * Lg / (ms_e2e / 1e3), "unit": "sequence-layers/s",
           "h2d_bytes_per_step": Lg * in_bytes, "d2h_bytes_per_step": Lg * out_bytes}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.profile:
        rate, n = gdn_oracle_rate(min(args.cpu_budget, 10.0), Lg)
        cpu = {"value": rate, "unit": "sequence-layers/s", "cores": 1, "kind": "oracle",
               "sample": f"{n} sequence-layers (one token, 32 heads of 128x128 state each), "
                         "float64 numpy oracle"}
    line = {
        "metric": "gdn_decode_sequence_layers_per_s", "value": value,
        "unit": "sequence-layers/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp32", "data": "synthetic",
        "config": {"workload": f"gdn_decode: {Lg} Gated DeltaNet layers x {B} sequences, "
                               f"{T} token(s) each", "Hk": s.Hk, "Hv": s.Hv, "dk": s.dk,
                   "dv": s.dv, "sequences": B, "tokens": T, "layers": Lg,
                   "parallelism": "replicas",
                   "l2": f"inputs larger than L2: {Lg * state_bytes / 1e9:.2f} GB of state "
                         "streamed per step"},
        "us_per_launch": us_launch,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / pk["hbm_gbs"], "traffic": measured_traffic(
                         "gdn_recurrence_kernel", f"gdn_B{B}_T{T}"),
                     "kernel": f"gdn_recurrence_kernel, {algo / 1e6:.1f} MB algorithmic per "
                               f"launch ({us_launch:.2f} us per launch)",
                     "peak_source": pk["source"]},
        "cpu_baseline": cpu, "e2e": e2e, "clocks": clk, "gpu_launches": args.steps * Lg,
        "parity_spot_check": parity,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


PHASES = [(0, "start"), (1, "input"), (25, "router_dots"), (2, "router"), (8, "logits_in"),
          (7, "sel_minmax"), (13, "sel_scan"), (14, "sel_cand"), (21, "rank"), (22, "certified"),
          (23, "slots"), (3, "select"), (24, "gu_first_task"), (9, "gu_tasks"), (4, "gateup"),
          (12, "h_exchange"), (5, "h_staged"), (10, "dn_data"), (20, "dn_first_task"),
          (16, "dn_tasks"), (11, "down"), (17, "y_written"), (18, "x_arrive"), (19, "sync"),
          (6, "end")]


def run_phases(args, wl):
    """Per-phase durations of the persistent decode kernel on a one-token stack:
    thread 0's SM cycle counter at each phase (an instrumented build of the
    library), median over CTAs and over the inner layers of the stack."""
    import torch

    import int4_routed_expert_decode_gb300 as moe
    from int4_routed_expert_decode_gb300 import build as moe_build
    here = os.path.join(ROOT, "int4_routed_expert_decode_gb300")
    moe.LIB_PATH = moe_build.build(defines=("MOE_DECODE_STAMPS",),
                                   lib_path=os.path.join(here, "_build", "stamps", "libmoe_stamps.so"),
                                   obj_dir=os.path.join(here, "_build", "stamps"))
    L = moe.lib()
    import ctypes
    L.moe_debug_stack_stamps.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    torch.cuda.set_device(0)
    NL = args.layers or 16
    layers = [moe.MoELayer(wl.E, wl.k, wl.H, wl.I, wl.Is, wl.G,
                           weights=synth.layer_weights(0, wl.wid, l, wl.shape), max_T=1)
              for l in range(NL)]
    norms = [torch.from_numpy(g.view(np.int16)).cuda().view(torch.bfloat16)
             for g in stack_norm_weights(wl, NL)]
    st = moe.MoEStack(layers, norms, STACK_EPS)
    xs = [torch.from_numpy(synth.tokens(0, wl.wid, 0, s, 1, wl.H)[0].view(np.int16)).cuda()
          .view(torch.bfloat16) for s in range(4)]
    for i in range(max(args.warmup, 3) + args.steps):
        st.forward(xs[i % 4])
    torch.cuda.synchronize()
    assert st.status() == moe.MOE_OK
    nC = torch.cuda.get_device_properties(0).multi_processor_count
    buf = np.zeros(NL * nC * 32, np.uint64)
    L.moe_debug_stack_stamps(st.stack, buf.ctypes.data, NL * nC * 32)
    a = buf.reshape(NL, nC, 32).astype(np.int64)
    clk = ClockSampler(0).start()  # the SM clock under the same load converts cycles to us
    t0 = time.perf_counter()
    i = 0
    while time.perf_counter() - t0 < 1.5:
        st.forward(xs[i % 4])
        i += 1
        if i % 32 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    mhz = clk.stop()["sm_mhz"] or 2070.0
    out = {"workload": wl.name, "layers": NL, "sm_mhz": mhz,
           "note": "us from the layer's start, per CTA (thread 0), median over CTAs and "
                   "layers 1..L-2; dn_* only on CTAs with a down tile", "phases": {}}
    for slot, name in PHASES:
        v = [(a[l, c, slot] - a[l, c, 0]) / mhz for l in range(1, NL - 1) for c in range(nC)
             if a[l, c, slot] and a[l, c, 0]]
        if v:
            out["phases"][name] = round(float(np.median(v)), 3)
    per = [np.median((a[l + 1, :, 0] - a[l, :, 0]) / mhz) for l in range(1, NL - 1)]
    out["layer_period_us"] = round(float(np.median(per)), 3)
    print(json.dumps(out), flush=True)
    st.close()


def main():
    args = parse()
    wl = synth.WORKLOADS[args.workload]
    if args.phases:
        run_phases(args, wl)
        return
    if args.mode == "gdn":
        run_gdn(args)
    elif args.impl == "reference":
        run_reference(args, wl)
    elif stack_mode(args, wl):
        run_ours_stack(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
