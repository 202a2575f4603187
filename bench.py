#!/usr/bin/env python
"""Benchmark of the MoE-layer forward megakernel on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload prefill]
                    [--mode persistent|multikernel|static] [--impl ours|reference]
                    [--residual-norm] [--option NAME=VALUE ...]

One step = one forward pass of the whole layer (router, top-k, permute,
gate/up + SiLU, down, combine) over one batch of synthetic tokens.  The default
workload is the large prefill layer (T=8192, d=7168, E=256 routed experts plus
one shared expert, k=8, f=2048): the largest of the five layer shapes, and the
one a per-layer throughput figure with no named configuration is read on.
The other shapes (tiny, decode, fine, skew) are selected with --workload.

Prints ONE JSON line (rank 0):
  value      tokens/s over all ranks, inputs resident in HBM, device-timed with
             CUDA events on the launching stream, L2 flushed between steps
             (outside the timed events)
  e2e        the same metric through moe_layer_forward_host: host->device copy
             of x, the forward, device->host copy of out, per step
  roofline   the megakernel against the measured HBM / bf16 peak
  cpu_baseline  the CPU oracle as it stands, on a bounded token sample
  clocks     nvidia-smi samples taken during the timed region
Multi-GPU (torchrun): every rank runs its own replica of the layer on its own
batch (the layer does not shard on one GPU: no collective on the data path);
value = all ranks' tokens / the slowest rank's time.

--impl reference times the CPU oracle (the only reference implementation this
method has) on the same workload and metric, one token per step.
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

REPO = os.path.dirname(os.path.abspath(__file__))
if REPO not in sys.path:
    sys.path.insert(0, REPO)

import numpy as np  # noqa: E402

import gen  # noqa: E402

METRIC = "MoE-layer tokens/s on 1 GB300; % of roofline (HBM or bf16 tensor peak)"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 512 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="prefill", choices=list(gen.WORKLOADS))
    ap.add_argument("--mode", default="persistent", choices=["persistent", "multikernel", "static"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--residual-norm", action="store_true",
                    help="time moe_layer_forward_residual_norm (residual add + RMSNorm fused "
                         "into the combine) instead of moe_layer_forward")
    ap.add_argument("--option", action="append", default=[], metavar="NAME=VALUE",
                    help="a layer option (MoELayer.set_option) for the timed runs")
    return ap.parse_args(argv)


# ---------------------------------------------------------------- environment

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def load_peaks():
    path = os.path.join(REPO, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(REPO, "persistent_megakernel_sm_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(name.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_from_profiles(workload: str, mode: str):
    """DRAM bytes per launch of the megakernel from the committed ncu summary,
    or None when there is none for the current kernel sources."""
    path = os.path.join(REPO, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        d = json.load(fh)
    ent = d.get(f"{workload}/{mode}")
    if not ent or ent.get("source_hash") != source_hash():
        return None
    return float(ent["dram_bytes_per_launch"])


def smi_device(dev: int) -> str:
    """nvidia-smi's id of CUDA device `dev` of this process: with
    CUDA_VISIBLE_DEVICES set, the entry it maps `dev` to (a physical index or a
    GPU UUID, both accepted by nvidia-smi -i); otherwise `dev` itself."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if 0 <= dev < len(ids):
            return ids[dev]
    return str(dev)


class ClockSampler:
    """nvidia-smi clock / throttle samples every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.lines = []
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", smi_device(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        if which == "start":
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        inside = [r for r in rows if self.t0 - 0.2 <= r[0] <= self.t1 + 0.2] or rows[-2:]
        sm = [float(p[1]) for _, p in inside if p[1].replace(".", "").isdigit()]
        mx = [float(p[2]) for _, p in inside if p[2].replace(".", "").isdigit()]
        pw = [float(p[3]) for _, p in inside if p[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for _, p in inside:
            for name, val in zip(names, p[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w": statistics.median(pw) if pw else None,
                "reasons": sorted(reasons), "samples": len(inside)}


def reduce_max(x: float, device: str) -> float:
    """Max of a per-rank scalar over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, ms_slowest: float, world: int) -> float:
    """Whole-job tokens/s: every rank's batch over the slowest rank's time."""
    return world * tokens_per_rank / (ms_slowest / 1e3)


# ---------------------------------------------------------------- workload facts

def algorithmic(w: gen.Workload, counts: np.ndarray):
    """Bytes and FLOPs one pass must move / do: weights of every expert that
    received a token (plus the shared expert and the router), x and out; the
    expert FLOPs 6 T (k + S) d f (router FLOPs 2 T d E reported apart)."""
    touched = int((counts > 0).sum()) + w.S
    wbytes = touched * 3 * w.f * w.d * 2 + w.E * w.d * 2
    io = 2 * w.T * w.d * 2
    flops = 6.0 * w.T * (w.k + w.S) * w.d * w.f
    return {"bytes": wbytes + io, "flops": flops, "router_flops": 2.0 * w.T * w.d * w.E,
            "touched_experts": touched}


# ---------------------------------------------------------------- our arm

def run_ours(args):
    import torch
    import persistent_megakernel_sm_gb300 as pkg

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    pkg.load_library()  # fails loudly when the CUDA library was not built

    w = gen.WORKLOADS[args.workload]
    inp = gen.make_inputs(w)

    def dev_bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()

    x = dev_bf16(inp["x"])
    wr = dev_bf16(inp["router_w"])
    wg = dev_bf16(inp["w_gate"])
    wu = dev_bf16(inp["w_up"])
    wd = dev_bf16(inp["w_down"])
    bias = None if inp["bias"] is None else torch.from_numpy(inp["bias"]).cuda()
    out = torch.empty((w.T, w.d), dtype=torch.bfloat16, device="cuda")
    layer = pkg.MoELayer(w.d, w.f, w.E, w.k, w.S)
    layer.reserve(w.T)
    layer.set_router_bias(bias)
    layer.set_option("mode", {"persistent": 0, "multikernel": 1, "static": 2}[args.mode])
    for kv in args.option:
        name, val = kv.split("=", 1)
        layer.set_option(name, int(val))
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    if args.residual_norm:  # seeded synthetic residual stream and norm weight
        g = torch.Generator(device="cpu").manual_seed(7)
        residual = (torch.randn((w.T, w.d), generator=g) * 0.8).to(torch.bfloat16).cuda()
        gamma = (1.0 + 0.25 * torch.randn(w.d, generator=g)).to(torch.bfloat16).cuda()
        norm_out = torch.empty_like(out)

        def fwd():
            layer.forward_residual_norm(x, wr, wg, wu, wd, residual, gamma, 1e-5, out, norm_out)
    else:
        def fwd():
            layer.forward(x, wr, wg, wu, wd, out)

    for _ in range(max(args.warmup, 3)):
        fwd()
    layer.check()
    counts = torch.empty(w.E, dtype=torch.int32, device="cuda")
    layer.get_routing(counts=counts)
    counts = counts.cpu().numpy()
    movers = layer.stat("mover_ctas")
    grid = layer.stat("grid")
    stolen = layer.stat("stolen")

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    sampler.mark("start")
    wall0 = time.perf_counter()
    for i in range(K):
        flush.zero_()
        ev[i][0].record(stream)
        fwd()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - wall0
    sampler.mark("stop")
    clocks = sampler.stop()
    rc = layer.status()
    if rc != 0:
        raise RuntimeError(f"device status {rc} during the timed region")
    times = [a.elapsed_time(b) for a, b in ev]
    ms = float(np.mean(times))
    ms_max = reduce_max(ms, "cuda")
    value = job_throughput(w.T, ms_max, world)

    # end to end through the host-buffer entry point
    e2e = None
    if not args.no_e2e:
        x_host = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).pin_memory()
        out_host = torch.empty((w.T, w.d), dtype=torch.bfloat16).pin_memory()
        for _ in range(3):
            layer.forward_host(w.T, x_host.data_ptr(), wr, wg, wu, wd, out_host.data_ptr())
        ke = min(args.e2e_steps, K)
        tot = 0.0
        for _ in range(ke):
            flush.zero_()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            layer.forward_host(w.T, x_host.data_ptr(), wr, wg, wu, wd, out_host.data_ptr())
            tot += time.perf_counter() - t0
        e2e_s = reduce_max(tot / ke, "cuda")
        e2e = {"value": job_throughput(w.T, e2e_s * 1e3, world), "unit": UNIT,
               "h2d_bytes_per_step": w.T * w.d * 2, "d2h_bytes_per_step": w.T * w.d * 2,
               "steps": ke, "ms_per_step": e2e_s * 1e3}

    peaks, peak_src = load_peaks()
    alg = algorithmic(w, counts)
    t = ms / 1e3
    t_hbm = alg["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_tc = alg["flops"] / (peaks["bf16_tflops"] * 1e12)
    traffic = traffic_from_profiles(args.workload, args.mode)
    if t_hbm >= t_tc:
        achieved = alg["bytes"] / t / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        achieved = alg["flops"] / t / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = traffic
    roof["peak_source"] = f"{peak_src} (burst figure: one launch per step, timed alone)"
    roof["kernel"] = {"persistent": "moe_persistent_kernel", "static": "moe_static_kernel",
                      "multikernel": "per-stage kernels (k_route .. k_combine), summed"}[args.mode]
    roof["timed"] = "forward call: one scheduler-reset memset + the kernel(s)"
    roof["algorithmic_bytes"] = alg["bytes"]
    roof["algorithmic_flops"] = alg["flops"]
    roof["roofline_frac"] = max(t_hbm, t_tc) / t

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, inp, args.cpu_seconds)

    kernels_per_step = 6 if args.mode == "multikernel" else 1
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {
            "workload": f"{w.name}: {w.describe()}", "T": w.T, "d": w.d, "E": w.E, "k": w.k,
            "f": w.f, "shared_experts": w.S, "mode": args.mode,
            "residual_rmsnorm": bool(args.residual_norm),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MB write, outside the timed events)",
            "inputs": "seeded synthetic (gen module), weights ~N(0,1/fan_in)",
            "mover_ctas": movers, "grid_ctas": grid, "stolen_tasks": stolen,
            "wall_s_timed_region": wall,
            "options": {kv.split("=", 1)[0]: int(kv.split("=", 1)[1]) for kv in args.option},
        },
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": kernels_per_step * K, "clocks": clocks,
        "us_per_layer": ms_max * 1e3, "ms_per_step_median": float(np.median(times)),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    layer.close()
    if world > 1:
        dist.destroy_process_group()


def cpu_baseline(w, inp, seconds):
    """The oracle as it stands (single-threaded C), one token at a time, until
    `seconds` of CPU work: tokens/s = tokens done / time."""
    import oracle
    wg, wu, wd = inp["w_gate"], inp["w_up"], inp["w_down"]
    rng = np.random.default_rng(7)
    order = rng.permutation(w.T)
    done = 0
    t0 = time.perf_counter()
    while True:
        t = int(order[done % w.T])
        oracle.layer(inp["x"], inp["router_w"], inp["bias"], wg, wu, wd, k=w.k, S=w.S,
                     tokens=np.array([t], dtype=np.int32))
        done += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": done / el, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{done} tokens of the {w.name} workload (routing + k experts"
                      f"{' + shared' if w.S else ''} per token), single-threaded C, fp64",
            "seconds": el}


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    w = gen.WORKLOADS[args.workload]
    inp = gen.make_inputs(w)
    import oracle
    rng = np.random.default_rng(11)
    order = rng.permutation(w.T)

    def step(i):
        t = int(order[i % w.T])
        oracle.layer(inp["x"], inp["router_w"], inp["bias"], inp["w_gate"], inp["w_up"],
                     inp["w_down"], k=w.k, S=w.S, tokens=np.array([t], dtype=np.int32))

    warm = 3  # untimed warm-up tokens: the contract's minimum, bounded (a token takes ~1 s)
    for i in range(warm):
        step(i)
    budget = 120.0
    done = 0
    t0 = time.perf_counter()
    while done < args.steps:
        step(done)
        done += 1
        if time.perf_counter() - t0 > budget:
            break
    el = time.perf_counter() - t0
    value = done / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": done, "warmup": warm, "ms_per_step": el / done * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.describe()}", "T": w.T, "d": w.d, "E": w.E,
                   "k": w.k, "f": w.f, "shared_experts": w.S,
                   "step": "one token of the batch (routing + its experts), CPU oracle",
                   "steps_requested": args.steps, "time_budget_s": budget},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{done} tokens of the {w.name} workload"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
