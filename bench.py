#!/usr/bin/env python3
"""Benchmark of the routed-MoE forward with per-token NVFP4 (one JSON line).

Workload (default): the decode-shaped layer - T=64 tokens, H=2048, E=128
experts, top-8, I=768 - run as a CUDA-graph replay of moe_forward.  One step
is one whole forward (router, top-k, permutation, quantization, both expert
GEMMs with their fused epilogues, finalize) over one batch of seeded
synthetic bf16 inputs resident in HBM.  L2 is flushed before every step,
outside the timed events: a 256 MB write, then a 256 MB read of another
buffer, so that the write-back of the flush's own dirty lines is not timed.

Run:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the layer has no exchange step); the value is all ranks' tokens over the
slowest rank's time.
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

METRIC = "MoE-layer tokens/s and % of roofline (FP4 tensor-core or HBM) at T=64/256/4096"
NVFP4_BYTES_PER_ELT = 0.5625      # 4-bit code + one E4M3 scale per 16 elements
STAGES = ("router", "topk", "permute", "quantize", "gemm_w13", "gemm_w2", "finalize")
SMALL_BATCH_TOKENS = 64           # the library's fused small-batch front end and atomic finalize


def kernels_per_forward(s, T, shared_inter=0):
    """Kernel launches of one forward: router, top-k, permute, quantize, w13,
    w2, finalize.  Up to 64 tokens: one fused front end, w13, the row
    requantization, w2, finalize (the bench runs per-token scales).  A shared
    expert adds its own stream's tile list, quantize, w13, w2, and up to 64
    tokens the row requantization between them."""
    shared = (5 if T <= SMALL_BATCH_TOKENS else 4) if shared_inter else 0
    return (7 if T > SMALL_BATCH_TOKENS else 5) + shared


def ordered_finalize(s, T):
    """Whether the forward stores bf16 (token, slot) rows and sums them in slot
    order (deterministic mode, and every forward above 64 tokens)."""
    return s.deterministic or T > SMALL_BATCH_TOKENS


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--config", default="c1_decode")
    p.add_argument("--tokens", type=int, default=None, help="override T of the workload")
    p.add_argument("--cpu-sample", type=int, default=4, help="tokens per oracle step")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--shared-inter", type=int, default=0,
                   help="add a shared expert of this intermediate width (0: routed experts only)")
    p.add_argument("--shared-average", action="store_true",
                   help="combine routed and shared outputs by their average instead of their sum")
    p.add_argument("--oracle-worker", action="store_true", help=argparse.SUPPRESS)
    return p.parse_args()


# --------------------------------------------------------------------------
# CPU oracle timing (runs in a single-threaded subprocess)
# --------------------------------------------------------------------------

def oracle_worker(args):
    import numpy as np

    import synthetic
    from oracle import moe as omoe
    from oracle import nvfp4 as onv

    wl = synthetic.make_workload(args.config, T=args.tokens)
    s = wl.shape
    n = min(args.cpu_sample, wl.T)
    tokens = np.linspace(0, wl.T - 1, n).astype(np.int64)
    x = omoe.as_f32(wl.x)
    wg = omoe.as_f32(wl.gate_w)
    bias = None if wl.bias is None else wl.bias.numpy()
    # weight conversion is load-time work (outside the forward), done untimed
    ids, _ = omoe.topk_route(omoe.router_logits(x[tokens], wg, bias), s.K)
    experts = np.unique(ids)
    E = s.E
    q13 = omoe.QuantWeights(np.zeros((E, 2 * s.I, s.H), np.uint8), np.zeros((E, 2 * s.I, s.H // 16), np.uint8),
                            np.ones(E, np.float32))
    q2 = omoe.QuantWeights(np.zeros((E, s.H, s.I), np.uint8), np.zeros((E, s.H, s.I // 16), np.uint8),
                           np.ones(E, np.float32))
    for e in experts:
        q13.codes[e], q13.sf[e], q13.gs[e] = onv.quantize_tensor(omoe.as_f32(wl.w13[e]))
        q2.codes[e], q2.sf[e], q2.gs[e] = onv.quantize_tensor(omoe.as_f32(wl.w2[e]))
    shared = None
    if args.shared_inter:
        w13s, w2s = synthetic.make_shared_weights(s, args.shared_inter)
        shared = (omoe.quantize_weights(omoe.as_f32(w13s)[None]), omoe.quantize_weights(omoe.as_f32(w2s)[None]))
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        omoe.moe_forward(x, wg, q13, q2, s.K, bias, tokens=tokens, shared=shared,
                         shared_average=args.shared_average)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    print(json.dumps({"tokens_per_step": int(n), "times": times, "experts": int(len(experts))}))


def run_oracle(args, steps, warmup):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-worker", "--config", args.config,
           "--steps", str(steps), "--warmup", str(warmup), "--cpu-sample", str(args.cpu_sample)]
    if args.tokens:
        cmd += ["--tokens", str(args.tokens)]
    if args.shared_inter:
        cmd += ["--shared-inter", str(args.shared_inter)] + (["--shared-average"] if args.shared_average else [])
    r = subprocess.run(cmd, capture_output=True, text=True, env=env)
    if r.returncode != 0:
        raise RuntimeError(f"oracle worker failed: {r.stderr[-2000:]}")
    d = json.loads(r.stdout.strip().splitlines()[-1])
    mean = statistics.mean(d["times"])
    return dict(value=d["tokens_per_step"] / mean, unit="tokens/s", cores=1, kind="oracle",
                sample=f"{d['tokens_per_step']} of the workload's tokens per step ({d['experts']} experts), "
                       f"{len(d['times'])} steps, forward only (weight conversion untimed), 1 thread",
                seconds_per_step=mean)


# --------------------------------------------------------------------------
# Clocks during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    """SM clock and clock-event reasons sampled while the timed loop runs.

    Reads NVML directly (libnvidia-ml through ctypes, read-only queries) every
    ~2 ms so that even a short timed region gets samples; falls back to
    nvidia-smi when NVML cannot be loaded.
    """

    NVML_CLOCK_SM = 1
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid=None, index=0, interval=0.002):
        import ctypes

        self.samples, self.reason_bits, self.max_mhz = [], 0, None
        self.stop_flag = threading.Event()
        self.lib = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            h = ctypes.c_void_p()
            ok = uuid and lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) == 0
            if not ok and lib.nvmlDeviceGetHandleByIndex_v2(int(index), ctypes.byref(h)) != 0:
                raise OSError("no NVML handle")
            self.lib, self.h = lib, h
            mx = ctypes.c_uint(0)
            if lib.nvmlDeviceGetMaxClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self.reason_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.thread = threading.Thread(target=self._loop, args=(interval,), daemon=True)
            self.thread.start()
        except (OSError, AttributeError):
            self.lib = None
            self.smi = _SmiSampler(uuid)

    def _loop(self, interval):
        import ctypes

        clk = ctypes.c_uint(0)
        rs = ctypes.c_ulonglong(0)
        while not self.stop_flag.is_set():
            if self.lib.nvmlDeviceGetClockInfo(self.h, self.NVML_CLOCK_SM, ctypes.byref(clk)) == 0:
                self.samples.append(float(clk.value))
            if self.reason_fn(self.h, ctypes.byref(rs)) == 0:
                self.reason_bits |= int(rs.value)
            time.sleep(interval)

    def stop(self):
        if self.lib is None:
            return self.smi.stop()
        self.stop_flag.set()
        self.thread.join(timeout=5)
        self.lib.nvmlShutdown()
        if not self.samples:
            return None
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(n for b, n in self.REASONS.items() if self.reason_bits & b),
                "samples": len(self.samples), "source": "nvml"}


class _SmiSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.rows = []
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if uuid:
            cmd += ["-i", uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 6:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if not self.rows:
            return None
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in self.rows:
            for name, v in zip(names, r[2:6]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(self.rows), "source": "nvidia-smi"}


# --------------------------------------------------------------------------
# Roofline helpers
# --------------------------------------------------------------------------

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# The sources that fix a GEMM launch's DRAM traffic: the kernel, its shared
# device helpers and argument block, and the host code that sizes its grid.
GEMM_SOURCES = ("common.cuh", "kernels.h", "kernels_gemm.cu", "moe_host.cu")


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "nvfp4_token_quantized_gb300", "csrc")
    for f in GEMM_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def dram_traffic(stage, config):
    """Per-launch DRAM bytes of a kernel from the committed ncu summary, or None
    when the kernel sources changed since those counters were taken."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    entry = d.get(config, {}).get(stage)
    if not entry or entry.get("source_hash") != kernel_source_hash():
        return None
    return entry.get("bytes_per_launch")


def stage_alg_bytes(s, T, touched):
    """Algorithmic bytes per launch of each stage (minimum traffic the stage's
    definition implies; NVFP4 operands at 0.5625 B per element)."""
    H, I, E, K = s.H, s.I, s.E, s.K
    R = T * K
    q = NVFP4_BYTES_PER_ELT
    return {
        "router": 2 * T * H + 2 * H * E + 4 * T * E,
        "topk": 4 * T * E + 8 * T * K,
        "permute": 4 * T * K + 16 * T * K,
        "quantize": 2 * T * H + q * R * H + 4 * R,
        "gemm_w13": touched * 2 * I * H * q + q * R * H + 4 * R + q * R * I + 4 * R,
        # ordered: the bf16 (token, slot) rows; atomic: the FP32 accumulator
        "gemm_w2": touched * H * I * q + q * R * I + 4 * R + (2 * R * H if ordered_finalize(s, T) else 4 * T * H),
        "finalize": (2 * R * H + 4 * R if ordered_finalize(s, T) else 4 * T * H) + 2 * T * H,
    }


def layer_alg_bytes(s, T, touched, shared_inter=0):
    # x in, out, router weight, and the NVFP4 weights of the experts that got
    # rows (and of the shared expert)
    return (2 * T * s.H + 2 * T * s.H + 2 * s.H * s.E
            + (touched * 3 * s.I + 3 * shared_inter) * s.H * NVFP4_BYTES_PER_ELT)


# --------------------------------------------------------------------------
# Our implementation
# --------------------------------------------------------------------------

def workload_config(s, T, world, shared_inter=0, shared_average=False):
    extra = {}
    shared_desc = ""
    if shared_inter:
        combine = "average" if shared_average else "sum"
        extra = {"shared_inter": shared_inter, "shared_combine": combine}
        shared_desc = f" + shared expert Is={shared_inter} ({combine}, second stream)"
    return {"workload": f"{s.name}: T={T} H={s.H} E={s.E} top-{s.K} I={s.I}{shared_desc}, CUDA-graph replay",
            "T": T, "H": s.H, "E": s.E, "top_k": s.K, "I": s.I, **extra,
            "finalize": ("ordered: bf16 (token, slot) rows summed in slot order" if ordered_finalize(s, T)
                         else "fp32 atomic in the w2 epilogue"),
            "l2": "flushed before every step outside the timed events: a 256 MB write, then a 256 MB read of "
                  "another buffer so the flush's own dirty lines are written back before timing (the weights, "
                  "338 MB at decode, also exceed L2)",
            "parallelism": f"replicas x{world}"}


def max_over_ranks(values, world):
    """Element-wise maximum of per-rank timings over all replicas (gloo group;
    no collective touches the data path)."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(v) for v in values], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


def replica_throughput(tokens_per_replica, world, ms_per_step):
    """Whole-job tokens/s: every replica processes its own batch each step, and
    the step time is the slowest replica's."""
    return tokens_per_replica * world / (ms_per_step / 1e3)


def run_ours(args, rank, world, local_rank):
    import torch

    import synthetic
    from nvfp4_token_quantized_gb300 import MoE, build

    build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = synthetic.make_workload(args.config, T=args.tokens)
    s = wl.shape
    T = wl.T
    Is = args.shared_inter
    layer = MoE(s.H, s.I, s.E, s.K, s.max_num_tokens, device=local_rank, deterministic=s.deterministic,
                shared_inter=Is, shared_average=args.shared_average)
    layer.load_weights(wl.w13.to(dev), wl.w2.to(dev))
    if Is:
        w13s, w2s = synthetic.make_shared_weights(s, Is)
        layer.load_shared_weights(w13s.to(dev), w2s.to(dev))
    x = wl.x.to(dev)
    gate_w = wl.gate_w.to(dev)
    bias = None if wl.bias is None else wl.bias.to(dev)
    out = torch.empty_like(x)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    evict = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def flush_l2(i):
        # write a buffer larger than L2, then read another one: L2 ends up
        # holding clean, unrelated lines, and the write-back of the flush's
        # dirty lines happens here rather than inside the timed step
        flush.fill_(i & 0xFF)
        evict.sum(dtype=torch.int32)

    # Two CUDA graphs of one forward (the decode path's serving mode): the
    # headline graph has no instrumentation; the second records an event at
    # every kernel boundary for the per-stage breakdown and the roofline of the
    # dominant kernel (the events serialise the kernels they separate).
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        layer.forward(x, gate_w, out=out, bias=bias)          # warm caches and lazy state
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        layer.forward(x, gate_w, out=out, bias=bias)
    layer.set_stage_timing(True)
    graph_staged = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_staged, stream=stream):
        layer.forward(x, gate_w, out=out, bias=bias)
    layer.set_stage_timing(False)
    torch.cuda.synchronize()

    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    for _ in range(args.warmup):
        flush_l2(1)
        graph.replay()
        flush_l2(2)
        graph_staged.replay()
    torch.cuda.synchronize()

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(uuid, index=local_rank)
    step_ms = []
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            flush_l2(i)
            start.record(stream)
            graph.replay()
            end.record(stream)
            end.synchronize()
            step_ms.append(start.elapsed_time(end))
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    total_ms = sum(step_ms)

    # per-stage breakdown (same inputs, instrumented graph)
    stages = {k: [] for k in STAGES}
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            flush_l2(i)
            graph_staged.replay()
            stream.synchronize()
            for k, v in layer.stage_times().items():
                stages[k].append(v)
    torch.cuda.synchronize()

    routing = layer.debug_routing()
    counts = torch.diff(routing["expert_offsets"]).cpu()
    touched = int((counts > 0).sum())

    # end to end through the host-buffer entry point (pinned host memory)
    xh = wl.x.pin_memory()
    gh = wl.gate_w.pin_memory()
    bh = None if wl.bias is None else wl.bias.pin_memory()
    oh = torch.empty_like(wl.x).pin_memory()
    for _ in range(max(1, args.warmup)):
        layer.forward_host(xh, gh, oh, bias=bh)
    e2e_s = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        layer.forward_host(xh, gh, oh, bias=bh)
        e2e_s.append(time.perf_counter() - t0)
    h2d = xh.numel() * 2 + gh.numel() * 2 + (0 if bh is None else bh.numel() * 4)
    d2h = oh.numel() * 2

    total_ms, e2e_total = max_over_ranks([total_ms, sum(e2e_s)], world)
    if rank != 0:
        layer.close()
        return None

    ms_per_step = total_ms / args.steps
    value = replica_throughput(T, world, ms_per_step)
    mean_stage = {k: statistics.mean(v) for k, v in stages.items() if v}
    dom = max(mean_stage, key=mean_stage.get)
    alg = stage_alg_bytes(s, T, touched)
    peak, peak_kind = measured_peaks()
    achieved = alg[dom] / (mean_stage[dom] / 1e3) / 1e9
    layer_bytes = layer_alg_bytes(s, T, touched, Is)
    layer_gbs = layer_bytes / (ms_per_step / 1e3) / 1e9
    result = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "nvfp4 (e2m1 x e2m1 with e4m3 block scales, fp32 accumulate)",
        "data": "synthetic (seeded bf16 N(0,1) activations, N(0,0.02) router/expert weights)",
        "config": workload_config(s, T, world, Is, args.shared_average),
        "roofline": {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": f"{peak_kind} hbm_gbs",
                     "alg_bytes_per_launch": alg[dom], "launch_ms": mean_stage[dom],
                     "traffic": dram_traffic(dom, s.name)},
        "layer_roofline": {"bound": "hbm", "alg_bytes": layer_bytes, "achieved_gbs": layer_gbs,
                           "frac": layer_gbs / peak, "touched_experts": touched},
        "stages_ms": mean_stage,
        "stages_note": "per-kernel times from an instrumented replay whose boundary events serialise the kernels",
        "e2e": {"value": T * world / (e2e_total / args.steps), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "path": "moe_forward_host (pinned host buffers, eager launches)"},
        "gpu_launches": kernels_per_forward(s, T, Is) * args.steps,
        "clocks": clk,
    }
    layer.close()
    return result


def main():
    args = parse()
    if args.oracle_worker:
        oracle_worker(args)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        r = run_oracle(args, args.steps, args.warmup)
        import synthetic

        s = synthetic.CONFIGS[args.config]
        line = {"impl": "reference", "metric": METRIC, "value": r["value"], "unit": "tokens/s", "n_gpus": 1,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["seconds_per_step"] * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
                "data": "synthetic", "config": workload_config(s, s.T if args.tokens is None else args.tokens, 1,
                                                          args.shared_inter, args.shared_average),
                "cpu_baseline": {k: r[k] for k in ("value", "unit", "cores", "kind", "sample")},
                "e2e": {"value": r["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("gloo", rank=rank, world_size=world)
    res = run_ours(args, rank, world, local_rank)
    if res is not None:
        if world == 1 and not args.no_cpu_baseline:
            cb = run_oracle(args, steps=10, warmup=1)
            res["cpu_baseline"] = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")}
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
