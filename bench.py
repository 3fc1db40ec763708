#!/usr/bin/env python
"""Throughput of the block-FP8 MoE layer (Drama 3 backbone shape) on GB300.

One step = one pass of the whole layer (router, quantisation, schedule,
routed experts, shared expert, combine) over one batch of synthetic rows.

At N=1 the workload is the one-row decode step (T=1, H=2048, 256 experts
top-8, I=Is=512, block-FP8 experts).  Weights are rotated over several
independent layer instances (0.77 GiB each, far above the 129 MB L2) so no
step finds its weights in L2.  The K timed steps run as CUDA graphs on one
stream; CUDA events bracket them.  With torchrun (N>1) every rank runs an
independent replica (rows are independent: weak scaling, no data-path
collective); the slowest rank's time counts.

Printed: one JSON line.  `--impl reference` times the CPU oracle instead.
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

METRIC = "MoE-layer rows/s"
UNIT = "rows/s"


PATHS = {"auto": 0, "prompt": 2, "chained": 3, "prompt_mma": 4, "rows": 6}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="decode_t1")
    ap.add_argument("--instances", type=int, default=16)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--rows", type=int, default=None,
                    help="rows per forward (default: the workload's); the 40-layer sweep "
                         "is quoted at 1, 4, 16, 64, 256 and 1024")
    ap.add_argument("--path", choices=tuple(PATHS), default="auto",
                    help="kernel path (MOE_OPT_PATH): auto picks by row count")
    ap.add_argument("--no-prompt", action="store_true",
                    help="leave out the prompt legs of the default one-row line")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ---- algorithmic bytes --------------------------------------------------------

def layer_bytes(s, T: int, U: int) -> int:
    """Bytes the layer must move: touched experts' e4m3 weights and scales,
    router, shared expert, gate vector, x and y."""
    G = s.group
    expert = 2 * s.inter * s.hidden + s.hidden * s.inter + \
        4 * ((2 * s.inter // G) * (s.hidden // G) + (s.hidden // G) * (s.inter // G))
    fixed = 4 * s.n_experts * s.hidden + 2 * (3 * s.shared_inter * s.hidden) + 2 * s.hidden
    return U * expert + fixed + 2 * 2 * T * s.hidden


def stage_bytes(s, T: int, U: int) -> dict:
    G, H, I, Is, E, k = s.group, s.hidden, s.inter, s.shared_inter, s.n_experts, s.top_k
    w13 = 2 * I * H + 4 * (2 * I // G) * (H // G)
    w2 = H * I + 4 * (H // G) * (I // G)
    # layer inputs, outputs and weights only: codes, SwiGLU rows, expert
    # outputs and other workspace traffic are not algorithmic bytes
    gateup = U * w13 + 2 * 2 * Is * H + 2 * T * H
    down = U * w2 + 2 * H * Is
    return {
        # decode path: one kernel for the whole layer
        "decode_row": layer_bytes(s, T, U),
        "decode_chain": layer_bytes(s, T, U),
        "decode_rows": layer_bytes(s, T, U),
        # decode path, chained variant (three kernels)
        "route_decode": 4 * E * H + 2 * T * H + 2 * H,
        "gateup_decode": gateup,
        "down_combine_decode": down + 2 * T * H,
        # prompt path
        "router": 4 * E * H + 2 * T * H,
        "quant_gamma": 2 * T * H + 2 * H,
        "topk": 0,
        "schedule": 0,
        "gateup": gateup,
        "down": down,
        "combine": 2 * T * H,
        # prompt path on tcgen05
        "router_tc": 4 * E * H + 2 * T * H,
        "quant_scatter": 2 * T * H + 2 * H,
        "shared_gateup_tc": 2 * 2 * Is * H + 2 * T * H,
        "gateup_tc": U * w13,
        "shared_down_tc": 2 * H * Is,
        "down_tc": U * w2,
    }


def stage_flops(s, T: int) -> dict:
    """Tensor-core flops of the GEMM stages, by the dtype their MMAs take."""
    H, I, Is, E, k = s.hidden, s.inter, s.shared_inter, s.n_experts, s.top_k
    return {
        "gateup_tc": ("fp8", 2 * T * k * 2 * I * H),
        "down_tc": ("fp8", 2 * T * k * H * I),
        "shared_gateup_tc": ("bf16", 2 * T * 2 * Is * H),
        "shared_down_tc": ("bf16", 2 * T * H * Is),
        "router_tc": ("bf16", 3 * 2 * T * E * H),
    }


def fp8_flops(s, T: int) -> int:
    return 2 * T * s.top_k * (2 * s.inter * s.hidden + s.hidden * s.inter)


# ---- clocks ------------------------------------------------------------------

QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, device_index: int):
        self.proc = None
        self.t0 = self.t1 = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={QUERY}", "--format=csv,noheader,nounits",
                 "-i", str(device_index), "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def finish(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.05)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            p = [v.strip() for v in line.split(",")]
            if len(p) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(p[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + p[0].split(".")[1]) if "." in p[0] else 0.0
                rows.append((ts + frac, p))
            except Exception:
                continue
        inside = [p for ts, p in rows if self.t0 is not None and self.t0 - 0.05 <= ts <= self.t1 + 0.05]
        use = inside if inside else [p for _, p in rows]
        sm = [float(p[2]) for p in use if p[2].replace(".", "").isdigit()]
        mx = [float(p[3]) for p in use if p[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in use for i in range(4) if p[6 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples_in_timed_region": len(inside),
                "power_w_max": max((float(p[4]) for p in use
                                    if p[4].replace(".", "").isdigit()), default=None)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("hbm_gbs"), d.get("bf16_tflops"), "measured"
    return 6800.0, 1900.0, "fallback"


def traffic_for(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu capture, or None once any of
    the kernel's source files has changed since (sha256 over them in order)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(f"{kernel}@{workload}")
    if not e:
        return None
    h = hashlib.sha256()
    for rel in e["sources"]:
        src = os.path.join(ROOT, rel)
        if not os.path.exists(src):
            return None
        with open(src, "rb") as f:
            h.update(f.read())
    if h.hexdigest() != e["sha256"]:
        return None
    return e["bytes_per_launch"]


# ---- the fused residual add + RMS norm + FP8 groups in front of the layer -----

ADDNORM_ROWS = {"addnorm_t1": 1, "addnorm_t11": 11, "addnorm_t1024": 1024}
ADDNORM_METRIC = "add-norm rows/s"


def addnorm_bytes(H: int, T: int) -> int:
    """Algorithmic bytes of one add-norm launch: read residual and x (bf16),
    write the new residual and the normed row (bf16), the codes (e4m3) and
    the group scales (fp32) of every row, plus gamma (bf16) once."""
    return T * (4 * 2 * H + H + 4 * (H // 128)) + 2 * H


def run_addnorm(args):
    import torch
    import torch.distributed as dist

    import block_fp8_mixture_router_gb300 as moe
    import workloads as W

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from block_fp8_mixture_router_gb300.build import build
    build()
    moe.load_library()
    s = W.FULL
    H = s.hidden
    T = args.rows if args.rows else ADDNORM_ROWS[args.workload]
    net = moe.MoELayer(moe.LayerShape(s.hidden, s.n_experts, s.top_k, s.inter, s.shared_inter,
                                      s.group), max_rows=1, device=local)
    # independent input sets (row blocks of one large draw) rotate so that
    # every launch reads from HBM: at least 512 MB pass per rotation
    per_set = addnorm_bytes(H, T)
    R = max(2, -(-(512 << 20) // per_set))
    r_all, x_all, g = W.make_addnorm(s, R * T, replica_seed(5000, rank), device=dev)
    h_all, xn_all = torch.empty_like(x_all), torch.empty_like(x_all)
    c_all = torch.empty((R * T, H), dtype=torch.uint8, device=dev)
    s_all = torch.empty((R * T, H // 128), dtype=torch.float32, device=dev)
    sets = [tuple(t[i * T:(i + 1) * T] if t is not g else g
                  for t in (r_all, x_all, g, h_all, xn_all, c_all, s_all)) for i in range(R)]
    ctx = net.ctx
    stream = torch.cuda.Stream(device=dev)

    def step(i):
        r, x, g, h, xn, c, sc = sets[i % R]
        rc = moe.moe_add_rmsnorm_quantize(ctx, r, x, g, W.NORM_EPS, T, h, xn, c, sc, stream)
        if rc != moe.MOE_OK:
            raise moe.MoEError(rc, "moe_add_rmsnorm_quantize")

    # about 0.3 s of launches, whole rotations (a launch takes at least ~2.5 us)
    est = max(2.5e-6, per_set / 5e12)
    K = args.steps if args.steps is not None else R * max(1, round(0.3 / est / R))
    Wm = max(3, args.warmup)
    with torch.cuda.stream(stream):
        for i in range(Wm):
            step(i)
    stream.synchronize()
    g_rot = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_rot, stream=stream):
        for i in range(R):
            step(i)
    full, rem = divmod(K, R)
    g_rem = None
    if rem:
        g_rem = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_rem, stream=stream):
            for i in range(rem):
                step(i)
    with torch.cuda.stream(stream):
        g_rot.replay()
    stream.synchronize()

    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if sampler:
        sampler.mark_start()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(full):
            g_rot.replay()
        if g_rem:
            g_rem.replay()
        e1.record(stream)
    e1.synchronize()
    if sampler:
        sampler.mark_end()
    torch.cuda.synchronize()
    ms = reduce_max(e0.elapsed_time(e1), dev)
    if world > 1:
        dist.barrier()
    clocks = sampler.finish() if sampler else None
    value = rows_per_second(world, K, T, ms / 1e3)
    try:
        quantiles = replay_quantiles(g_rot, stream, R, full)
    except Exception as e:  # reported, never fatal to the line
        quantiles = {"unavailable": f"{type(e).__name__}: {e}"[:200]}
    hbm, _, peak_kind = measured_peaks()
    launch_us = ms / K * 1e3
    ab = addnorm_bytes(H, T)
    gbs = ab / (launch_us * 1e-6) / 1e9
    line = {
        "metric": ADDNORM_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": Wm, "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "rows": T, "hidden": H, "eps": W.NORM_EPS,
                   "inputs": "residual N(0,1), block output N(0,0.25), gamma 1 + N(0,0.01), bf16",
                   "l2": f"inputs rotate over {R} independent row blocks "
                         f"({R * per_set / 2**20:.0f} MiB per rotation) > 129 MB L2",
                   "timing": "CUDA graphs of whole rotations, CUDA events on the launch stream",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "kernel": "add_rmsnorm_quant", "achieved": gbs, "peak": hbm,
                     "unit": "GB/s", "frac": gbs / hbm, "peak_kind": peak_kind,
                     "algorithmic_bytes_per_launch": ab, "avg_launch_us": launch_us,
                     "duration_source": "CUDA events over the timed region (one launch per step)",
                     "traffic": traffic_for("add_rmsnorm_quant", args.workload)},
        "gpu_launches": K,
        "clocks": clocks,
        "step_ms_quantiles": quantiles,
    }

    # end to end: residual and x from pinned host memory, all four outputs back
    r, x, g, h, xn, c, sc = sets[0]
    rh, xh = r.cpu().pin_memory(), x.cpu().pin_memory()
    outs_h = [t.cpu().pin_memory() for t in (h, xn, c, sc)]
    Ke = min(K, 2000)

    def e2e_step():
        with torch.cuda.stream(stream):
            r.copy_(rh, non_blocking=True)
            x.copy_(xh, non_blocking=True)
            step(0)
            for dst, src in zip(outs_h, (h, xn, c, sc)):
                dst.copy_(src, non_blocking=True)
        stream.synchronize()

    for _ in range(3):
        e2e_step()
    t0 = time.perf_counter()
    for _ in range(Ke):
        e2e_step()
    et = reduce_max(time.perf_counter() - t0, dev)
    line["e2e"] = {"value": rows_per_second(world, Ke, T, et), "unit": UNIT,
                   "h2d_bytes_per_step": 2 * T * H * 2,
                   "d2h_bytes_per_step": T * (2 * H * 2 + H + 4 * (H // 128)),
                   "steps": Ke, "api": "moe_add_rmsnorm_quantize, host copies per step"}
    if rank == 0 and world == 1:
        v, n = cpu_addnorm(r.cpu(), x.cpu(), g.cpu(), args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": f"{n} oracle rows of input set 0 ({args.workload}), "
                                          f"{args.cpu_seconds:.0f} s budget"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    net.close()
    if world > 1:
        dist.destroy_process_group()


def cpu_addnorm(r, x, g, budget_s: float):
    """The oracle's add-norm, one row at a time, for about budget_s seconds."""
    import oracle
    import workloads as W
    oracle.build()
    rb, xb, gb = W.bf16_bits(r), W.bf16_bits(x), W.bf16_bits(g)
    rows = 0
    t0 = time.perf_counter()
    while rows == 0 or time.perf_counter() - t0 < budget_s:
        i = rows % rb.shape[0]
        oracle.add_rmsnorm(rb[i:i + 1], xb[i:i + 1], gb, W.NORM_EPS)
        rows += 1
    return rows / (time.perf_counter() - t0), rows


def reference_addnorm(args):
    rank, _, _ = dist_env()
    if rank != 0:
        return
    import workloads as W
    T = args.rows if args.rows else ADDNORM_ROWS[args.workload]
    r, x, g = W.make_addnorm(W.FULL, T, replica_seed(5000, 0))
    steps = args.steps if args.steps is not None else 5
    budget = min(60.0, args.cpu_seconds)
    t0 = time.perf_counter()
    v, n = cpu_addnorm(r, x, g, budget / steps)
    for _ in range(steps - 1):
        cpu_addnorm(r, x, g, budget / steps)
    dt = time.perf_counter() - t0
    line = {
        "impl": "reference", "metric": ADDNORM_METRIC, "value": v, "unit": UNIT,
        "n_gpus": args.gpus, "steps": steps, "warmup": 0, "ms_per_step": 1e3 * dt / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": args.workload, "rows": T, "hidden": W.FULL.hidden},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"the oracle's add-norm row by row, {budget:.0f} s in all"},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---- the layer taking the residual stream: fused add-norm vs two calls -------

ADDNORM_LAYER_ROWS = {"addnorm_layer_t1": 1, "addnorm_layer_t11": 11,
                      "addnorm_layer_t1024": 1024}


def run_addnorm_layer(args):
    """moe_forward_addnorm (the add-norm inside the layer's launches) against
    moe_add_rmsnorm_quantize followed by moe_forward, on the same rotation of
    layer instances; the line's value is the fused call's rows/s."""
    import torch
    import torch.distributed as dist

    import block_fp8_mixture_router_gb300 as moe
    import workloads as W

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from block_fp8_mixture_router_gb300.build import build
    build()
    moe.load_library()
    s = W.FULL
    H = s.hidden
    T = args.rows if args.rows else ADDNORM_LAYER_ROWS[args.workload]
    L = max(1, args.instances if T < 64 else 2)
    shape = moe.LayerShape(s.hidden, s.n_experts, s.top_k, s.inter, s.shared_inter, s.group)
    nets, ins, outs = [], [], []
    for i in range(L):
        seed = replica_seed(1 + 7919 * i, rank)
        net = moe.MoELayer(shape, max_rows=max(T, 16), device=local)
        net.load(W.make_layer(s, seed, device=dev))
        nets.append(net)
        r, x, g = (t.to(dev) for t in W.make_addnorm(s, T, replica_seed(5000 + i, rank)))
        ins.append((r, x, g))
        outs.append(tuple(torch.empty_like(x) for _ in range(3)) +
                    (torch.empty((T, H), dtype=torch.uint8, device=dev),
                     torch.empty((T, H // 128), dtype=torch.float32, device=dev)))
    stream = torch.cuda.Stream(device=dev)

    def fused(i):
        j = i % L
        r, x, g = ins[j]
        h, xn, y, _, _ = outs[j]
        rc = moe.moe_forward_addnorm(nets[j].ctx, r, x, g, W.NORM_EPS, T, h, None, y, stream)
        if rc != moe.MOE_OK:
            raise moe.MoEError(rc, "moe_forward_addnorm")

    def separate(i):
        j = i % L
        r, x, g = ins[j]
        h, xn, y, c, sc = outs[j]
        rc = moe.moe_add_rmsnorm_quantize(nets[j].ctx, r, x, g, W.NORM_EPS, T, h, xn, c, sc,
                                          stream)
        if rc == moe.MOE_OK:
            rc = moe.moe_forward(nets[j].ctx, xn, y, T, stream)
        if rc != moe.MOE_OK:
            raise moe.MoEError(rc, "add-norm then forward")

    K = args.steps if args.steps is not None else max(L, 32000 // T)
    Wm = max(3, args.warmup)
    res = {}
    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    if sampler:
        sampler.mark_start()
    for name, fn in (("fused", fused), ("separate", separate)):
        with torch.cuda.stream(stream):
            for i in range(Wm):
                fn(i)
        stream.synchronize()
        g_k = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_k, stream=stream):
            for i in range(K):
                fn(i)
        g_warm = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_warm, stream=stream):
            for i in range(L):
                fn(i)
        with torch.cuda.stream(stream):
            g_k.replay()
        stream.synchronize()
        if world > 1:
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        warm_gpu(stream)
        with torch.cuda.stream(stream):
            for _ in range(max(1, int(30e-3 / max(1e-6, 15e-6 * L * max(1, T // 16))))):
                g_warm.replay()
            e0.record(stream)
            g_k.replay()
            e1.record(stream)
        e1.synchronize()
        ms = reduce_max(e0.elapsed_time(e1), dev)
        res[name] = {"value": rows_per_second(world, K, T, ms / 1e3), "ms_per_step": ms / K}
    if sampler:
        sampler.mark_end()
    clocks = sampler.finish() if sampler else None
    f, sp = res["fused"], res["separate"]
    line = {
        "metric": "MoE-layer rows/s (residual add + RMS norm + layer)", "value": f["value"],
        "unit": UNIT, "n_gpus": world, "steps": K, "warmup": Wm, "ms_per_step": f["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic",
        "config": {"workload": args.workload, "rows": T, "hidden": H, "eps": W.NORM_EPS,
                   "layer_instances": L,
                   "l2": f"weights rotate over {L} layer instances > 129 MB L2",
                   "timing": "CUDA graphs of K steps, CUDA events on the launch stream",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "separate": {"value": sp["value"], "ms_per_step": sp["ms_per_step"],
                     "api": "moe_add_rmsnorm_quantize then moe_forward"},
        "saved_us_per_step": (sp["ms_per_step"] - f["ms_per_step"]) * 1e3,
        "saved_bytes_per_step": T * H * 2 * 2,  # the normed rows written and read again
        # one launch per fused step at one row; more rows launch the add-norm
        # kernel and the forward's kernels (not counted here)
        "gpu_launches": K if T == 1 else None,
        "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    for net in nets:
        net.close()
    if world > 1:
        dist.destroy_process_group()


# ---- replicas ---------------------------------------------------------------

def reduce_max(value: float, dev=None) -> float:
    """The largest value over all ranks (the value itself without a process
    group): the slowest replica's time counts."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64,
                     device=dev if dev is not None else torch.device("cpu"))
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_seed(seed: int, rank: int) -> int:
    """Each replica draws its own layers and rows (independent work)."""
    return seed + 104729 * rank


def rows_per_second(world: int, steps: int, rows_per_step: int, seconds: float) -> float:
    """Whole-job throughput: every replica processed steps x rows_per_step."""
    return world * steps * rows_per_step / seconds


# ---- reference arm: the CPU oracle -----------------------------------------

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import torch  # noqa: F401
    import oracle
    import workloads as W
    wl = W.WORKLOADS[args.workload]
    s = wl.shape
    T = args.rows if args.rows else wl.rows
    seed = W.layer_seed(wl, 0) if wl.layers > 1 else wl.seed
    oracle.build()
    # a bounded sample of the workload: up to two of its rows per step, and
    # at most about a minute of steps in all
    sample = max(1, min(T, 2))
    x = W.make_x(s, sample, seed, wl.x_kind)
    wr = W.make_router(s, seed, wl.x_kind)
    idx = set()
    xb = W.bf16_bits(x)
    for r in range(xb.shape[0]):
        idx |= set(oracle.router_row(xb[r], wr.numpy(), s.top_k)[1].tolist())
    layer = W.to_numpy_layer(W.make_layer(s, seed, wl.x_kind, experts=sorted(idx)))
    steps_req = args.steps if args.steps is not None else 5
    if args.warmup:
        oracle.moe_rows(layer, xb[:1])
    budget_s = 60.0
    steps = 0
    t0 = time.perf_counter()
    while steps < steps_req and (steps == 0 or time.perf_counter() - t0 < budget_s):
        oracle.moe_rows(layer, xb)
        steps += 1
    dt = time.perf_counter() - t0
    rows = steps * xb.shape[0]
    value = rows / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": steps, "warmup": 1 if args.warmup else 0, "ms_per_step": 1e3 * dt / steps,
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "rows": T, "hidden": s.hidden,
                   "experts": s.n_experts, "top_k": s.top_k, "inter": s.inter,
                   "shared_inter": s.shared_inter},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{steps} oracle passes of {xb.shape[0]} of the {T} rows "
                                   f"of {wl.name} (steps capped at about {budget_s:.0f} s)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---- our arm -----------------------------------------------------------------

def cpu_baseline(layer_host, xb, budget_s: float):
    import oracle
    oracle.build()
    rows = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        r = rows % xb.shape[0]
        oracle.moe_rows(layer_host, xb[r:r + 1])
        rows += 1
    dt = time.perf_counter() - t0
    return rows / dt, rows


def replay_quantiles(graph, stream, steps_per_replay: int, replays: int,
                     cap: int = 200) -> dict:
    """p10 / median / p90 of the time per step (ms), from CUDA events recorded
    on the launch stream between consecutive replays of the timed graph
    (after the timed region, so the events do not touch it)."""
    import torch
    n = min(cap, replays)
    if n < 3 or graph is None:
        return {"unavailable": "fewer than 3 whole-graph replays"}
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for i in range(n):
            graph.replay()
            ev[i + 1].record(stream)
    ev[-1].synchronize()
    per = sorted(ev[i].elapsed_time(ev[i + 1]) / steps_per_replay for i in range(n))
    return {"p10": per_quantile(per, 0.1), "median": per_quantile(per, 0.5),
            "p90": per_quantile(per, 0.9), "replays": n,
            "steps_per_replay": steps_per_replay}


def per_quantile(sorted_vals, q: float) -> float:
    """Linear-interpolated quantile of an ascending list."""
    pos = q * (len(sorted_vals) - 1)
    lo = int(pos)
    hi = min(lo + 1, len(sorted_vals) - 1)
    return sorted_vals[lo] + (sorted_vals[hi] - sorted_vals[lo]) * (pos - lo)


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def cpu_baseline_threads(layer_host, xb, budget_s: float, threads: int):
    """The same oracle with its rows spread over `threads` host threads, the
    per-row code unchanged.  The oracle is a C library behind ctypes, which
    lets go of the GIL for the length of each call, so the threads run side by
    side; one call first builds the oracle's e4m3 table, which is read-only
    afterwards."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    oracle.build()
    oracle.moe_rows(layer_host, xb[:1])
    counts = [0] * threads
    t0 = time.perf_counter()

    def worker(i):
        n = 0
        while n == 0 or time.perf_counter() - t0 < budget_s:
            r = (i + n * threads) % xb.shape[0]
            oracle.moe_rows(layer_host, xb[r:r + 1])
            n += 1
        counts[i] = n

    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(worker, range(threads)))
    dt = time.perf_counter() - t0
    return sum(counts) / dt, sum(counts)


def warm_gpu(stream):
    """Keep the GPU busy for ~50 us on `stream` so that the host enqueues the
    timed region's start event and graphs while the device is still working:
    the region then starts when its first step starts, not when the host
    catches up."""
    import torch
    with torch.cuda.stream(stream):
        torch.cuda._sleep(100_000)


def measure_layer(moe, W, wl, T: int, K: int, Wm: int, L: int, path: str, dev, rank: int,
                  world: int, e2e_steps: int = 2000) -> dict:
    """Builds L layer instances (or wl's chained layers), times exactly K
    steps of T rows in CUDA graphs, and returns the line's measured fields."""
    import torch
    s = wl.shape
    local = dev.index
    sweep = wl.layers > 1
    L = wl.layers if sweep else L
    shape = moe.LayerShape(s.hidden, s.n_experts, s.top_k, s.inter, s.shared_inter, s.group)
    nets, xs, ys, layers = [], [], [], []
    for i in range(L):
        seed = replica_seed(W.layer_seed(wl, i) if sweep else wl.seed + 7919 * i, rank)
        layer = W.make_layer(s, seed, wl.x_kind, device=dev)
        net = moe.MoELayer(shape, max_rows=max(T, 16), device=local)
        net.load(layer)
        net.set_option(moe.MOE_OPT_PATH, PATHS[path])
        nets.append(net)
        if not sweep or i == 0:
            xs.append(W.make_x(s, T, seed, wl.x_kind, device=dev))
        ys.append(torch.empty((T, s.hidden), dtype=torch.bfloat16, device=dev))
        if i == 0:
            layers.append(layer)
        del layer
    torch.cuda.synchronize()
    stream = torch.cuda.Stream(device=dev)
    layers_per_step = L if sweep else 1
    if sweep:
        # the layers as one chain: y of layer j is the input of layer j + 1
        # (one launch over all layers at one row)
        chain = moe.MoEChain(nets)
        y_all = torch.empty((L, T, s.hidden), dtype=torch.bfloat16, device=dev)
        ys = [y_all[j] for j in range(L)]

    def step(i):
        if sweep:
            chain.forward(xs[0], y_all, stream=stream)
            return
        j = i % L
        nets[j].forward(xs[j], ys[j], stream=stream)

    with torch.cuda.stream(stream):
        for i in range(Wm):
            step(i)
    stream.synchronize()

    def capture(n, first=0):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(first, first + n):
                step(i)
        return g

    # the K timed steps: whole graphs of up to `chunk` steps (a multiple of
    # the rotation), then the remainder; K <= chunk is one graph
    per_rot = 1 if sweep else L
    chunk = max(per_rot, (max(1, 4096 // (launches_hint(T) * layers_per_step)) // per_rot) * per_rot)
    full, rem = divmod(K, chunk)
    g_full = capture(chunk) if full else None
    g_rem = capture(rem, full * chunk) if rem else None
    g_warm = g_rem if g_rem is not None else g_full
    t0w = torch.cuda.Event(enable_timing=True)
    t1w = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        if g_full:
            g_full.replay()
        t0w.record(stream)
        g_warm.replay()
        t1w.record(stream)
    stream.synchronize()
    # untimed replays right before the timed region keep the GPU busy (and
    # its clocks up) for ~30 ms after the idle sampler start-up
    n_warm = max(1, min(2000, int(30.0 / max(t0w.elapsed_time(t1w), 1e-3))))

    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if sampler:
        sampler.mark_start()
    warm_gpu(stream)
    with torch.cuda.stream(stream):
        for _ in range(n_warm):
            g_warm.replay()
        e0.record(stream)
        for _ in range(full):
            g_full.replay()
        if g_rem:
            g_rem.replay()
        e1.record(stream)
    e1.synchronize()
    if sampler:
        sampler.mark_end()
    torch.cuda.synchronize()
    ms = reduce_max(e0.elapsed_time(e1), dev)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    clocks = sampler.finish() if sampler else None
    value = rows_per_second(world, K, T * layers_per_step, ms / 1e3)
    # spread per step: replays of one rotation's graph after the timed region
    try:
        g_q = capture(per_rot)
        quantiles = replay_quantiles(g_q, stream, per_rot, max(3, min(200, 4000 // per_rot)))
    except Exception as e:  # reported, never fatal to the line
        quantiles = {"unavailable": f"{type(e).__name__}: {e}"[:200]}

    # per-kernel device times (events after every launch), same rotation
    stage_ms = {}
    P = min(64, max(8, L * 4))
    for i in range(P):
        j = 0 if sweep else i % L
        for name, t in nets[j].profile(xs[j], ys[j], stream=stream):
            stage_ms.setdefault(name, []).append(t)
    chain_one_launch = sweep and T == 1
    if chain_one_launch:
        # one launch of the one-row kernel over every layer: the per-layer
        # time comes from the timed region
        stage_ms = {"decode_chain": [ms / K / layers_per_step]}
    stage_avg = {n: sum(v) / len(v) for n, v in stage_ms.items()}
    stage_prof = dict(stage_avg)
    launches_per_step = sum(STAGE_LAUNCHES.get(n, 1) for n in stage_avg)
    duration_source = "per-kernel CUDA events of a profiled forward (moe_profile_forward)"
    if len(stage_avg) == 1:
        # one stage per layer forward: its launches are the timed region's
        # launches, so their average duration is the timed region's
        stage_avg = {n: ms / K / layers_per_step for n in stage_avg}
        duration_source = ("CUDA events over the timed region (one launch over all "
                           "layers, per layer)" if chain_one_launch else
                           "CUDA events over the timed region (one launch per layer forward)")

    # touched experts per layer instance; in the sweep each layer's input is
    # the previous layer's output (ys[j - 1] after the timed steps)
    Us = []
    for j in range(L):
        src = (xs[0] if j == 0 else ys[j - 1]) if sweep else xs[j]
        idx, _ = nets[j].route(src, stream=stream)
        stream.synchronize()
        Us.append(len(set(idx.cpu().numpy().ravel().tolist())))
    U = sum(Us) / len(Us)
    sb = stage_bytes(s, T, U)
    hbm, bf16_tf, peak_kind = measured_peaks()
    dom = max(stage_avg, key=stage_avg.get)
    dom_gbs = sb[dom] / (stage_avg[dom] * 1e-3) / 1e9
    # the binding roof of the dominant kernel: bytes at HBM speed, or its
    # tensor-core flops at the peak of its dtype (fp8 = 2 x the bf16 peak)
    sf = stage_flops(s, T).get(dom)
    roof = {"bound": "hbm", "kernel": dom, "achieved": dom_gbs, "peak": hbm, "unit": "GB/s",
            "frac": dom_gbs / hbm, "peak_kind": peak_kind, "algorithmic_bytes_per_launch": sb[dom],
            "avg_launch_us": stage_avg[dom] * 1e3, "duration_source": duration_source,
            "traffic": traffic_for(dom, wl.name)}
    if sf is not None:
        tf_peak = bf16_tf * (2.0 if sf[0] == "fp8" else 1.0)
        tf = sf[1] / (stage_avg[dom] * 1e-3) / 1e12
        roof["tensor_tflops"] = tf
        roof["tensor_peak"] = tf_peak
        roof["tensor_dtype"] = sf[0]
        if sf[1] / (tf_peak * 1e12) > sb[dom] / (hbm * 1e9):
            roof.update({"bound": "tensor", "achieved": tf, "peak": tf_peak, "unit": "TFLOP/s",
                         "frac": tf / tf_peak,
                         "peak_kind": peak_kind + (" (bf16 x 2 for fp8)" if sf[0] == "fp8" else "")})
    lb = layer_bytes(s, T, U)
    step_ms = ms / K / layers_per_step  # per layer
    out = {
        "value": value, "ms_per_step": ms / K, "steps": K, "warmup": Wm,
        "layer_instances": L, "layers_per_step": layers_per_step,
        "l2": (f"{L} chained layers, {L * lb / 2**30:.1f} GiB touched per step"
               if sweep else
               f"weights rotate over {L} layer instances "
               f"({L * lb / 2**30:.1f} GiB touched per rotation)") + " > 129 MB L2",
        "roofline": roof,
        "layer_roofline": {"bound": "hbm", "algorithmic_bytes_per_step": lb,
                           "achieved": lb / (step_ms * 1e-3) / 1e9, "peak": hbm, "unit": "GB/s",
                           "frac": lb / (step_ms * 1e-3) / 1e9 / hbm,
                           "distinct_experts": U,
                           "fp8_tflops": fp8_flops(s, T) / (step_ms * 1e-3) / 1e12,
                           "fp8_frac": fp8_flops(s, T) / (step_ms * 1e-3) / 1e12
                           / (2.0 * bf16_tf)},
        "stages_us": {n: round(v * 1e3, 3) for n, v in stage_prof.items()},
        "step_ms_quantiles": quantiles,
        "gpu_launches": K if chain_one_launch else K * launches_per_step * layers_per_step,
        "clocks": clocks,
    }

    # end to end through the C ABI with host buffers (copies inside the timed region)
    xh = [x.cpu().pin_memory() for x in xs]
    yh = [torch.empty_like(v).pin_memory() for v in xh]
    Ke = max(1, min(K, e2e_steps))

    def e2e_step(i):
        if sweep:  # one copy in, the layers on the device, one copy out
            with torch.cuda.stream(stream):
                xd = xh[0].to(dev, non_blocking=True)
                chain.forward(xd, y_all, stream=stream)
                yh[0].copy_(y_all[L - 1], non_blocking=True)
            stream.synchronize()
            return
        j = i % L
        nets[j].forward_host(xh[j], yh[j], stream=stream)

    # untimed: every layer instance once
    for i in range(max(3, L)):
        e2e_step(i)
    t0 = time.perf_counter()
    for i in range(Ke):
        e2e_step(i)
    et = reduce_max(time.perf_counter() - t0, dev)
    out["e2e"] = {"value": rows_per_second(world, Ke, T * layers_per_step, et), "unit": UNIT,
                  "h2d_bytes_per_step": T * s.hidden * 2, "d2h_bytes_per_step": T * s.hidden * 2,
                  "steps": Ke,
                  "api": "moe_chain_forward over the layers, host copies per step" if sweep
                  else "moe_forward_host"}
    out["_host"] = (W.to_numpy_layer(layers[0]), W.bf16_bits(xs[0]))
    if sweep:
        chain.close()
    for net in nets:
        net.close()
    del nets, xs, ys, layers
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


# stages that time more than one launch (none today: moe_profile_forward
# records one event after every launch)
STAGE_LAUNCHES = {}


def launches_hint(T: int) -> int:
    """Kernel launches of one forward of T rows (graph size bound only)."""
    return 1 if T <= 4 else 12


# prompt legs reported beside the one-row headline: (workload, steps, instances)
PROMPT_LEGS = (("prompt_t1024", 50, 2), ("prompt_t16384", 20, 1))


def run_ours(args):
    import torch
    import torch.distributed as dist

    import block_fp8_mixture_router_gb300 as moe
    import workloads as W

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from block_fp8_mixture_router_gb300.build import build
    build()
    moe.load_library()

    wl = W.WORKLOADS[args.workload]
    s = wl.shape
    T = args.rows if args.rows else wl.rows
    layers_per_step = wl.layers if wl.layers > 1 else 1
    K = args.steps if args.steps is not None else max(1, 32000 // (T * layers_per_step))
    K = max(1, K)
    Wm = max(3, args.warmup)
    r = measure_layer(moe, W, wl, T, K, Wm, max(1, args.instances), args.path, dev, rank, world)
    host, xb = r.pop("_host")
    line = {
        "metric": METRIC, "value": r["value"], "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": Wm, "ms_per_step": r["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
        "config": {"workload": wl.name, "rows": T, "hidden": s.hidden, "experts": s.n_experts,
                   "top_k": s.top_k, "inter": s.inter, "shared_inter": s.shared_inter,
                   "activations": "bf16", "expert_weights": "e4m3, fp32 128x128 block scales",
                   "layer_instances": r["layer_instances"],
                   "layers_per_step": r["layers_per_step"], "l2": r["l2"],
                   "timing": "CUDA graphs of whole steps, CUDA events on the launch stream",
                   "kernel_path": args.path,
                   "parallelism": "replicas" if world > 1 else "single GPU"},
    }
    for key in ("roofline", "layer_roofline", "stages_us", "step_ms_quantiles", "gpu_launches",
                "clocks", "e2e"):
        line[key] = r[key]

    # the prompt path beside the one-row headline: its own legs, each with
    # its own roofline (FP8 tensor roof where the flops bind), stages and e2e
    if args.workload == "decode_t1" and not args.rows and not args.no_prompt:
        legs = {}
        for name, steps, inst in PROMPT_LEGS:
            pw = W.WORKLOADS[name]
            try:
                pr = measure_layer(moe, W, pw, pw.rows, steps, Wm, inst, "auto", dev, rank,
                                   world, e2e_steps=20)
                pr.pop("_host")
                pr["workload"] = name
                pr["rows"] = pw.rows
                pr["unit"] = UNIT
                legs[name] = pr
            except Exception as e:  # reported, never fatal to the headline
                legs[name] = {"unavailable": f"{type(e).__name__}: {e}"[:300]}
        line["prompt"] = legs

    if rank == 0 and world == 1:
        v, n = cpu_baseline(host, xb, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": f"{n} single-row passes of layer instance 0 "
                                          f"({wl.name}), {args.cpu_seconds:.0f} s budget"}
        # the same oracle over every host core the process may use
        nt = host_threads()
        if nt > 1:
            bt = min(args.cpu_seconds, 6.0)
            try:
                v2, n2 = cpu_baseline_threads(host, xb, bt, nt)
                line["cpu_baseline_all_cores"] = {
                    "value": v2, "unit": UNIT, "cores": nt, "kind": "oracle",
                    "sample": f"{n2} single-row passes of layer instance 0 ({wl.name}) on "
                              f"{nt} threads, {bt:.0f} s budget"}
            except Exception as e:  # reported, never fatal to the line
                line["cpu_baseline_all_cores"] = {"unavailable": f"{type(e).__name__}: {e}"[:200]}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.workload in ADDNORM_ROWS:
        (reference_addnorm if args.impl == "reference" else run_addnorm)(args)
    elif args.workload in ADDNORM_LAYER_ROWS:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the add-norm layer leg has no oracle timing; see the layer and "
                              "add-norm workloads"}), flush=True)
        else:
            run_addnorm_layer(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
