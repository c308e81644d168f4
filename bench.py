"""Benchmark of the NVFP4 W4A16 sigmoid-top-k MoE decode layer on GB300.

One step = one decode step through every MoE layer of a Flint-shaped model:
47 distinct layers (49 layers, the first two dense; "vLLM Day-0 support for
Recursive's Flint", "Flint model architecture"), T tokens each, captured into
one CUDA graph.  Metric: per-layer decode time and effective HBM GB/s over the
bytes a layer must read (router, the selected experts and the shared expert,
x and out).  The selected bytes are counted from the ids each layer returns.
Distinct layers make every step read ~1 GB at T=1, far more than L2 (126 MB),
so nothing is served from L2 across layers.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload flint1]
  python bench.py --impl reference ...   (the CPU oracle, timed as the reference arm)

Rank 0 prints one JSON line.  Under torchrun every rank runs its own layers
(weak scaling, no collective on the data path) and the timed region is the
max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer decode µs & effective HBM GB/s (selected-expert bytes) at T=1/8"
WORKLOADS = {
    # name: (config index, layers per step)
    "flint1": (1, 47),
    "flint8": (2, 47),
    "ml4": (4, 6),
    "zipf64": (3, 16),
    "tiny": (0, 64),
    "ml4fp8s": (5, 6),        # ML4 with its FP8 block-scaled shared expert
    "inkling": (6, 2),        # Inkling-2-Small-shaped, NVFP4 experts
    "inkling_mx8": (7, 2),    # the same with MXFP8 experts
    "flint_mx4": (8, 47),     # Flint-shaped, MXFP4 experts
    "inkling_w4a4": (9, 2),   # Inkling-2-Small-shaped, W4A4 (Four-Over-Six activations)
    "zipf64_w4a4": (10, 16),  # Zipf-routed Flint-shaped T=64, W4A4
}

# DRAM bytes (read + write) per launch of the single-launch kernel, from one
# ncu capture per workload (summaries under profiles/), valid only for the
# kernel source they were taken on: reported as `traffic` while fused.cu
# hashes to the value below, null otherwise.  (The value below is that of a
# source that differs from the captured one, 3fd6c6f8882e58a0, in its header
# comment only.)
NCU_TRAFFIC = {
    "flint1": {"bytes": 20788736, "fused_cu_sha256_16": "6c9876c1b570cbb2"},
    "flint8": {"bytes": 124420864, "fused_cu_sha256_16": "6c9876c1b570cbb2"},
}

def ncu_traffic(workload: str):
    import hashlib
    rec = NCU_TRAFFIC.get(workload)
    if not rec:
        return None
    with open(os.path.join(ROOT, "nvfp4_weight_only_fp32_gb300", "csrc", "fused.cu"), "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()[:16]
    return rec["bytes"] if sha == rec["fused_cu_sha256_16"] else None


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0, help="timed steps (0: enough for ~1.5 s)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="flint1", choices=sorted(WORKLOADS))
    ap.add_argument("--layers", type=int, default=0, help="override layers per step")
    ap.add_argument("--secondary", default="flint8", help="second workload reported in the line ('' = none)")
    ap.add_argument("--extras", default="ml4,zipf64,zipf64-gemv,tiny,ml4fp8s,inkling,inkling_mx8,flint_mx4,"
                                        "inkling_w4a4,zipf64_w4a4,flint1-coop,flint8-coop",
                    help="further workloads timed and reported under 'workloads' ('' = none); "
                         "a '-gemv' suffix turns the grouped kernels off, '-coop' launches the single "
                         "launch as a cooperative grid, '-chain' runs the three-kernel chain instead")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--grouped-min", type=int, default=0,
                    help="grouped_min_tokens of the layers (0: library default, -1: GEMV kernels only)")
    ap.add_argument("--score-func", default="sigmoid", choices=["sigmoid", "softmax"],
                    help="routing score of the measured workload's layers (softmax: the chain)")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append((time.time(), ln.strip()))

    def stop(self, t0: float | None = None, t1: float | None = None):
        """Median SM clock and throttle reasons over the samples taken between
        wall-clock times t0 and t1 (the timed region)."""
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, ln in self.lines:
            if t0 is not None and not (t0 <= ts <= t1):
                continue
            f = [v.strip() for v in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples in the timed region"],
                    "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU)
# ---------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_init(ws, backend):
    if ws > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)
        return dist
    return None


def max_over_ranks(value: float, dist, device=None) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, dist, device=None) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ---------------------------------------------------------------------------
# CPU oracle leg (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------
def oracle_sample(cfg_index: int, seconds: float, seed: int, want_out: bool = False, threads: int = 0):
    """Time the oracle on whole-layer forwards of the workload until `seconds`
    of CPU work have run (threads: 0 = all host cores).
    -> dict(value GB/s, per_layer_s, layers, cores, ...)."""
    import numpy as np
    import gen
    import oracle
    c = gen.config(cfg_index)
    router = gen.make_router(c, seed)
    x = gen.make_x(c, seed)
    ids, *_ = oracle.route({"cfg": c, **router}, x)
    layer = {"cfg": c, **router, **gen.make_experts(c, seed, np.unique(ids))}
    nthreads = threads if threads > 0 else oracle.max_threads()
    pairs = c["T"] * (c["k"] + c["S"])
    cores = min(nthreads, pairs)
    n, t0, res = 0, time.perf_counter(), None
    while True:
        res = oracle.forward(layer, x, nthreads=nthreads)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds or n >= 10000:
            break
    U = len(np.unique(res[2]))
    b = gen.selected_bytes(c, U)
    out = {"value": b * n / el / 1e9, "per_layer_s": el / n, "layers": n, "cores": cores,
           "selected_bytes": b, "seconds": el}
    if want_out:
        out["layer"], out["x"], out["result"] = layer, x, res
    return out


def run_reference(args):
    ws, rank, local = dist_env()
    if rank != 0:
        return 0
    ci, _ = WORKLOADS[args.workload]
    import gen
    c = gen.config(ci)
    if args.steps <= 0:
        args.steps = 3        # each step is a bounded sample of CPU work
    per_step = max(1.0, args.cpu_seconds / max(1, args.steps))
    for w in range(args.warmup):
        oracle_sample(ci, 0.0, gen.BASE_SEED + 100 + w)
    total_b, layers, cores, el = 0.0, 0, 1, 0.0
    for k in range(args.steps):
        r = oracle_sample(ci, per_step, gen.BASE_SEED + 200 + k)
        total_b += r["selected_bytes"] * r["layers"]
        layers += r["layers"]
        cores = r["cores"]
        el += r["seconds"]     # oracle work only; input generation is not timed
    gbs = total_b / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{c['name']}: T={c['T']} H={c['H']} E={c['E']} top-{c['k']} "
                               f"I={c['I']} +{c['S']} shared, one layer per sample",
                   "step": f"about {per_step:.1f} s of whole-layer oracle forwards"},
        "us_per_layer": el * 1e6 / max(1, layers),
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{layers} whole-layer FP64 forwards of the {c['name']} workload"},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU leg
# ---------------------------------------------------------------------------
class Chain:
    """L distinct layers of one workload on the current GPU."""

    def __init__(self, moe, torch, gen, ci, L, seed0, grouped_min=0, score_func="sigmoid", fused=0):
        self.c = gen.config(ci, score_func=score_func)
        c = self.c
        self.T, self.L = c["T"], L
        self.layers, self.xs, self.outs, self.ids, self.ws = [], [], [], [], []
        for l in range(L):
            lay = gen.make_layer_torch(c, seed0 + l)
            self.layers.append(moe.MoELayer(lay, max_tokens=self.T, grouped_min_tokens=grouped_min, fused=fused))
            del lay
            self.xs.append(gen.make_x_torch(c, seed0 + l))
            self.outs.append(torch.empty((self.T, c["H"]), dtype=torch.bfloat16, device="cuda"))
            self.ids.append(torch.empty((self.T, c["k"]), dtype=torch.int32, device="cuda"))
            self.ws.append(torch.empty((self.T, c["k"]), dtype=torch.float32, device="cuda"))
        torch.cuda.synchronize()

    def enqueue(self, moe, stage=None):
        for l in range(self.L):
            h = self.layers[l].h
            if stage is None:
                moe.moe_decode_forward(h, self.xs[l], self.T, self.outs[l], self.ids[l], self.ws[l])
            elif stage == "route":
                moe.moe_stage_route(h, self.xs[l], self.T, self.ids[l], self.ws[l])
            elif stage == "gate_up":
                moe.moe_stage_gate_up(h, self.xs[l], self.T)
            elif stage == "down":
                moe.moe_stage_down(h, self.T, self.outs[l])

    def close(self):
        for lay in self.layers:
            lay.close()


def capture(torch, fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        fn()
    torch.cuda.synchronize()
    return g


def time_graph(torch, g, stream, warmup, steps, sampler=None, clock_pass_steps=0):
    """CUDA-event time of `steps` replays after `warmup` untimed ones.  With a
    sampler, clocks are sampled from the start of an untimed pass of
    `clock_pass_steps` replays of the same graph (long enough for the 200 ms
    sampler, run just before) through the end of the timed region."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    tc = None
    if sampler:
        sampler.start()
        time.sleep(0.3)
        tc = time.time()
        with torch.cuda.stream(stream):
            for _ in range(clock_pass_steps):
                g.replay()
    t0 = time.time()
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(steps):
            g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    clocks = None
    if sampler:
        clocks = sampler.stop(tc, t1)
        clocks["window"] = (f"{clock_pass_steps} untimed replays of the same graph just before the timed "
                            f"region ({t0 - tc:.2f} s), then the timed region ({t1 - t0:.3f} s)")
    return e0.elapsed_time(e1), clocks


def auto_steps(torch, g, stream, warmup, target_s=1.5):
    """Timed steps for a ~target_s timed region (so that the clock sampler,
    at 200 ms, sees it), from a short calibration after the warm-up."""
    ms, _ = time_graph(torch, g, stream, warmup, 3)
    return int(min(20000, max(20, target_s * 1e3 / max(ms / 3, 1e-3))))


def byte_counts(gen, chain, np):
    """Selected bytes per layer from the ids each layer returned, plus the
    gate/up kernel's algorithmic bytes (weights of the slots, x in, h out)."""
    c = chain.c
    T, H, I, Is, S, k = c["T"], c["H"], c["I"], c["Is"], c["S"], c["k"]
    sel, gu, Us = [], [], []
    for l in range(chain.L):
        U = len(np.unique(chain.ids[l].cpu().numpy()))
        Us.append(U)
        sel.append(gen.selected_bytes(c, U))
        w13 = U * (2 * I * H // 2 + 2 * I * H // 16 + 8) + S * (2 * Is * H // 2 + 2 * Is * H // 16 + 8)
        gu.append(w13 + T * H * 2 + T * (k + S) * max(I, Is) * 2)
    return sel, gu, Us


def run_gpu(args):
    import numpy as np
    import torch
    import gen
    import nvfp4_weight_only_fp32_gb300 as moe
    from nvfp4_weight_only_fp32_gb300 import build as moe_build

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = dist_init(ws, "nccl")
    moe_build.build()
    moe.lib()
    dev = torch.device("cuda", local)
    peak, peak_kind = peaks()
    ci, L = WORKLOADS[args.workload]
    L = args.layers or L
    seed0 = gen.BASE_SEED + 1000 * (rank + 1) + 100 * ci
    chain = Chain(moe, torch, gen, ci, L, seed0, args.grouped_min, args.score_func)
    c = chain.c
    stream = torch.cuda.Stream()

    g_full = capture(torch, lambda: chain.enqueue(moe), stream)
    sel, gu_bytes, Us = byte_counts(gen, chain, np)
    long_steps = auto_steps(torch, g_full, stream, args.warmup)     # ~1.5 s of replays
    if args.steps <= 0:
        args.steps = long_steps
        if dist is not None:
            args.steps = int(max_over_ranks(float(args.steps), dist, dev))
    barrier(dist)
    sampler = ClockSampler(local)
    ms, clocks = time_graph(torch, g_full, stream, args.warmup, args.steps, sampler,
                            clock_pass_steps=long_steps if args.steps < long_steps else 0)
    barrier(dist)
    ms_max = max_over_ranks(ms, dist, dev)
    bytes_step = float(sum(sel))
    total_bytes = sum_over_ranks(bytes_step * args.steps, dist, dev)
    value = total_bytes / (ms_max * 1e-3) / 1e9
    us_layer = ms * 1e3 / (args.steps * L)

    # per-stage graphs of the three-kernel chain: each kernel's average launch
    # duration (the chain is what moe_decode_forward runs when the single
    # launch does not apply)
    stage_us = {}
    for st in ("route", "gate_up", "down"):
        g = capture(torch, lambda st=st: chain.enqueue(moe, st), stream)
        sms, _ = time_graph(torch, g, stream, 3, max(5, args.steps // 2))
        stage_us[st] = sms * 1e3 / (max(5, args.steps // 2) * L)
        del g
    single = chain.layers[0].info().single_launch_max_tokens >= chain.T
    if single:
        # one fused_kernel launch per layer: the timed graph is nothing but
        # those launches, so its per-layer time is the launch duration
        rk_name, rk_bytes, rk_us = "fused_kernel (single launch)", float(np.mean(sel)), us_layer
    else:
        rk_name, rk_bytes, rk_us = "gemv_kernel<gate/up>", float(np.mean(gu_bytes)), stage_us["gate_up"]
    achieved = rk_bytes / (rk_us * 1e-6) / 1e9

    # end to end through the host-buffer entry point (pinned memory): x up,
    # the layer, its output down (the routing ids and weights are optional
    # outputs of that call, not requested here)
    T, H, k = c["T"], c["H"], c["k"]
    xh = [chain.xs[l].cpu().pin_memory() for l in range(L)]
    oh = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(L)]

    def e2e_step():
        for l in range(L):
            moe.moe_decode_forward_host(chain.layers[l].h, xh[l], T, oh[l], None, None, stream)

    # the step's host-buffer calls captured once into a CUDA graph, as a
    # decode loop runs them: every replay moves x up (a copy, or at one or
    # two tokens the kernel's own reads of the pinned rows) and the output
    # down (the kernels' stores into the pinned rows); eager calls if capture
    # is refused
    try:
        g_e2e = capture(torch, e2e_step, stream)
        e2e_run, e2e_mode = g_e2e.replay, "CUDA graph of the host-buffer calls"
    except Exception:
        torch.cuda.synchronize()
        g_e2e, e2e_run, e2e_mode = None, e2e_step, "eager host-buffer calls"
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            e2e_run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            e2e_run()
    e1.record(stream)
    torch.cuda.synchronize()
    del g_e2e
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)
    e2e_total = sum_over_ranks(bytes_step * args.steps, dist, dev)
    e2e = {"value": e2e_total / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
           "h2d_bytes_per_step": L * T * H * 2,
           "d2h_bytes_per_step": L * T * H * 2,
           "us_per_layer": e2e_ms * 1e3 / (args.steps * L), "mode": e2e_mode}
    # cold single-layer latency: one call of the first layer right after
    # writing a scratch buffer of twice the L2 size (its weights, x and the
    # code's data are then not in L2), median of a few tries
    scratch = torch.empty(2 * torch.cuda.get_device_properties(dev).L2_cache_size // 4 + 1024,
                          dtype=torch.float32, device=dev)
    cold = []
    for i in range(7):
        with torch.cuda.stream(stream):
            scratch.fill_(float(i))
            e0.record(stream)
            moe.moe_decode_forward(chain.layers[0].h, chain.xs[0], T, chain.outs[0], chain.ids[0], chain.ws[0],
                                   stream)
            e1.record(stream)
        torch.cuda.synchronize()
        cold.append(e0.elapsed_time(e1) * 1e3)
    del scratch
    cold_us = sorted(cold)[len(cold) // 2]
    chain.close()
    del chain, g_full
    torch.cuda.empty_cache()

    def other(name, grouped_min=0, fused=0):
        """Per-layer time of another workload: its own distinct layers in one
        CUDA graph, timed like the main one (same warm-up and step count)."""
        oi, oL = WORKLOADS[name]
        ch2 = Chain(moe, torch, gen, oi, oL, seed0 + 50000 + 1000 * oi, grouped_min, fused=fused)
        g2 = capture(torch, lambda: ch2.enqueue(moe), stream)
        sel2, _, U2 = byte_counts(gen, ch2, np)
        st2 = max(args.steps, 5)
        ms2, _ = time_graph(torch, g2, stream, args.warmup, st2)
        us2 = ms2 * 1e3 / (st2 * oL)
        b2 = float(np.mean(sel2))
        c2 = ch2.c
        one = ch2.layers[0].info().single_launch_max_tokens >= ch2.T
        res = {"workload": f"{c2['name']}: T={c2['T']} H={c2['H']} E={c2['E']} top-{c2['k']} "
                           f"I={c2['I']} +{c2['S']} shared, experts {c2['efmt']}, shared {c2['sfmt']}, "
                           + ("W4A4 Four-Over-Six activations, " if c2.get("w4a4") else "")
                           + f"{oL} layers per step",
               "us_per_layer": us2, "GBps": b2 / (us2 * 1e-6) / 1e9,
               "frac_of_measured": b2 / (us2 * 1e-6) / 1e9 / peak,
               "selected_bytes_per_layer": b2, "unique_experts_mean": float(np.mean(U2)),
               "path": ("single launch" + (", cooperative grid" if fused > 0 else "")) if one else
                       ("chain" + (", grouped kernels off" if grouped_min < 0 else
                                   (", grouped tensor-core kernels for slots of >= 8 tokens"
                                    if c2["T"] > 8 and "fp8" not in c2["efmt"] + c2["sfmt"] else ""))),
               "steps": st2}
        ch2.close()
        del g2
        torch.cuda.empty_cache()
        return res

    secondary = None
    workloads = {}
    if rank == 0:
        if args.secondary not in ("", "none") and args.secondary != args.workload:
            secondary = other(args.secondary)
        for name in [w for w in args.extras.split(",") if w and w != "none"]:
            # "-gemv": the grouped kernels off; "-coop": the single launch as a
            # cooperative grid; "-chain": the three-kernel chain, no single launch
            base = name.rsplit("-", 1)[0] if name.endswith(("-gemv", "-coop", "-chain")) else name
            if name == base == args.workload:
                continue
            fused = 1 if name.endswith("-coop") else (-1 if name.endswith("-chain") else 0)
            workloads[name] = other(base, -1 if name.endswith("-gemv") else 0, fused)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        r = oracle_sample(ci, args.cpu_seconds, gen.BASE_SEED + 7)
        r1 = oracle_sample(ci, max(2.0, args.cpu_seconds / 4), gen.BASE_SEED + 8, threads=1)
        cpu = {"value": r["value"], "unit": "GB/s", "cores": r["cores"], "kind": "oracle",
               "sample": f"{r['layers']} whole-layer FP64 forwards of one {c['name']} layer "
                         f"(T={c['T']}), {r['seconds']:.1f} s",
               "us_per_layer": r["per_layer_s"] * 1e6,
               "single_thread": {"value": r1["value"], "unit": "GB/s", "cores": 1,
                                 "us_per_layer": r1["per_layer_s"] * 1e6,
                                 "sample": f"{r1['layers']} forwards, {r1['seconds']:.1f} s"}}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "w4a16(e2m1*e4m3 x bf16->f16 mma, fp32 acc)",
            "data": "synthetic",
            "config": {"workload": f"{c['name']}: T={c['T']} H={c['H']} E={c['E']} top-{c['k']} "
                                   f"I={c['I']} +{c['S']} shared"
                                   + ("" if args.score_func == "sigmoid" else f", {args.score_func} routing"),
                       "layers_per_step": L, "tokens_per_layer": c["T"],
                       "l2": f"inputs larger than L2: {L} distinct layers, "
                             f"{bytes_step / 1e6:.0f} MB selected bytes per step",
                       "graph": "one CUDA graph per step; " + ("one single-launch kernel per layer" if single else
                                                                       "3 kernels per layer chained with PDL")},
            "us_per_layer": us_layer,
            "cold_us_per_layer": cold_us,
            "selected_bytes_per_layer": bytes_step / L,
            "unique_experts_mean": float(np.mean(Us)),
            "frac_of_8TBps": value / 8000.0,
            "chain_stage_us": stage_us,
            "roofline": {"bound": "hbm", "kernel": rk_name, "achieved": achieved,
                         "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": ncu_traffic(args.workload) if single else None,
                         "peak_kind": f"{peak_kind} (copy bandwidth, burst)",
                         "algorithmic_bytes_per_launch": rk_bytes, "launch_us": rk_us},
            "clocks": clocks,
            "e2e": e2e,
            "gpu_launches": (1 if single else 3) * L * args.steps,
            "cpu_baseline": cpu,
        }
        if secondary:
            line["secondary"] = secondary
        if workloads:
            line["workloads"] = workloads
        print(json.dumps(line), flush=True)
    barrier(dist)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
