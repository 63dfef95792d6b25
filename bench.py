#!/usr/bin/env python3
"""Benchmark of the routed-MoE forward with per-token NVFP4 (one JSON line).

The metric is quoted at T = 64, 256 and 4096 tokens.  With no flags one run
times all three on the layer H=2048, E=128 experts, top-8, I=768:

* headline: the prefill chunk, T=4096 on an instance created for 4096 tokens
  (the tensor-core throughput workload and the largest single-GPU one);
* per_config: the decode batch (T=64) and the speculative-decode batch
  (T=256, Zipf-skewed routing, deterministic mode).

One step is one whole forward (router, top-k, permutation, quantization,
both expert GEMMs with their fused epilogues, finalize) over one batch of
seeded synthetic bf16 inputs resident in HBM, run as a CUDA-graph replay.
L2 is flushed before every step, outside the timed events: a 256 MB write,
then a 256 MB read of another buffer, so that the write-back of the flush's
own dirty lines is not timed.  ms_per_step is the median over the timed steps.

Run:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                      [--config all|c1_decode|c2_specdecode|c3_prefill|c4_stress]
Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the layer has no exchange step); the value is all ranks' tokens over the
slowest rank's time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s and % of roofline (FP4 tensor-core or HBM) at T=64/256/4096"
NVFP4_BYTES_PER_ELT = 0.5625      # 4-bit code + one E4M3 scale per 16 elements
STAGES = ("router", "topk", "permute", "quantize", "gemm_w13", "gemm_w2", "finalize")
SMALL_BATCH_TOKENS = 64           # the library's fused small-batch front end and atomic finalize
HEADLINE = "c3_prefill"           # T = 4096: the tensor-core throughput workload
PER_CONFIG = ("c1_decode", "c2_specdecode")
# Dense FP4 tensor-core peak relative to dense bf16 (nominal 13.5 / 2.25
# PFLOP/s): the FP4 peak is the measured bf16 peak times this ratio.
FP4_OVER_BF16 = 6.0


def kernels_per_forward(s, T, shared_inter=0):
    """Kernel launches of one forward: router, top-k, permute, quantize, w13,
    w2, finalize.  Up to 64 tokens: one fused front end, w13, w2, finalize,
    plus the row requantization kernel unless nearly every expert gets a row
    (T*K >= 4E: the w13 GEMM then requantizes in its own tail; the bench runs
    per-token scales).  A shared expert adds its own stream's tile list,
    quantize, w13, w2, and up to 64 tokens the row requantization between
    them."""
    shared = (5 if T <= SMALL_BATCH_TOKENS else 4) if shared_inter else 0
    if T > SMALL_BATCH_TOKENS:
        return 7 + shared
    all_experts = T * s.K >= 4 * s.E
    return (4 if all_experts else 5) + shared


def ordered_finalize(s, T):
    """Whether the forward stores bf16 (token, slot) rows and sums them in slot
    order (deterministic mode, and every forward above 64 tokens)."""
    return s.deterministic or T > SMALL_BATCH_TOKENS


def parse(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--config", default="all",
                   help="'all' (headline T=4096 prefill plus the T=64 and T=256 workloads) or one workload name")
    p.add_argument("--tokens", type=int, default=None, help="override T of a single workload")
    p.add_argument("--cpu-sample", type=int, default=None,
                   help="tokens per oracle process per step (default: 4 for the baseline leg, 1 for --impl reference)")
    p.add_argument("--cpu-procs", type=int, default=0,
                   help="oracle processes for the all-cores baseline (0: every core of the affinity mask, at most 16)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--shared-inter", type=int, default=0,
                   help="add a shared expert of this intermediate width (0: routed experts only)")
    p.add_argument("--shared-average", action="store_true",
                   help="combine routed and shared outputs by their average instead of their sum")
    p.add_argument("--accurate-sigmoid", action="store_true",
                   help="SwiGLU with sigmoid 1/(1+expf(-g)) instead of the hardware-tanh form")
    return p.parse_args(argv)


# --------------------------------------------------------------------------
# Workloads (weights drawn once per layer shape and seed, shared by the
# workloads that have the same layer)
# --------------------------------------------------------------------------

_WEIGHTS = {}


def workload(name, T=None):
    import synthetic

    s = synthetic.CONFIGS[name]
    key = (s.E, s.H, s.I, 0)
    if key not in _WEIGHTS:
        _WEIGHTS[key] = synthetic.make_weights(s, seed=0)
    w13, w2 = _WEIGHTS[key]
    x = synthetic.make_activations(s, T=T, seed=0)
    bias = synthetic.zipf_router_bias(s, seed=0) if s.zipf_bias else None
    return synthetic.Workload(shape=s, x=x, gate_w=synthetic.make_router(s, seed=0), w13=w13, w2=w2, bias=bias)


# --------------------------------------------------------------------------
# CPU oracle timing: P single-threaded processes, each running the oracle's
# forward on its own tokens of the workload, started together
# --------------------------------------------------------------------------

def affinity():
    try:
        cpus = sorted(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        cpus = list(range(os.cpu_count() or 1))
    return cpus


def _ranges(cpus):
    out, start, prev = [], None, None
    for c in cpus:
        if start is None:
            start = prev = c
        elif c == prev + 1:
            prev = c
        else:
            out.append(f"{start}-{prev}" if prev != start else f"{start}")
            start = prev = c
    if start is not None:
        out.append(f"{start}-{prev}" if prev != start else f"{start}")
    return ",".join(out)


def _oracle_quantize(args):
    """Worker: oracle quantization of one expert's two weight tensors."""
    import numpy as np

    from oracle import nvfp4 as onv

    w13_bits, w2_bits = args
    f = lambda b: (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)
    return onv.quantize_tensor(f(w13_bits)), onv.quantize_tensor(f(w2_bits))


def _oracle_proc(path, tokens, steps, warmup, top_k, shared_average, barrier, queue):
    """One timed oracle process: untimed set-up (the quantized weights are
    memory-mapped), a start barrier shared with the other processes, then
    warmup + steps forwards of its tokens."""
    import numpy as np

    from oracle import moe as omoe

    x = np.load(os.path.join(path, "x.npy"), mmap_mode="r")
    wg = np.load(os.path.join(path, "wg.npy"))
    bias = np.load(os.path.join(path, "bias.npy")) if os.path.exists(os.path.join(path, "bias.npy")) else None
    q = [omoe.QuantWeights(np.load(os.path.join(path, f"{n}_codes.npy"), mmap_mode="r"),
                           np.load(os.path.join(path, f"{n}_sf.npy"), mmap_mode="r"),
                           np.load(os.path.join(path, f"{n}_gs.npy"))) for n in ("w13", "w2")]
    shared = None
    if os.path.exists(os.path.join(path, "s13_codes.npy")):
        shared = tuple(omoe.QuantWeights(np.load(os.path.join(path, f"{n}_codes.npy")),
                                         np.load(os.path.join(path, f"{n}_sf.npy")),
                                         np.load(os.path.join(path, f"{n}_gs.npy"))) for n in ("s13", "s2"))
    xs = np.asarray(x[np.asarray(tokens)], dtype=np.float32)
    barrier.wait()
    times = []
    for i in range(warmup + steps):
        t0 = time.perf_counter()
        omoe.moe_forward(xs, wg, q[0], q[1], top_k, bias, shared=shared, shared_average=shared_average)
        dt = time.perf_counter() - t0
        if i >= warmup:
            times.append(dt)
    queue.put((len(tokens), times))


def run_oracle(wl, steps, warmup, per_proc, procs, shared=None, shared_average=False):
    """The oracle, as it stands, on the host cores: `procs` single-threaded
    processes (spawned, each pinned to nothing), each on per_proc tokens of
    the workload per step; throughput = the sum over processes of their
    tokens / their mean step time (they run concurrently).  The experts the
    sampled tokens route to are quantized beforehand (load-time work, untimed,
    in a spawn pool)."""
    import multiprocessing as mp

    import numpy as np

    from oracle import moe as omoe

    s = wl.shape
    n = min(procs * per_proc, wl.T)
    procs = max(1, min(procs, n))
    tokens = np.linspace(0, wl.T - 1, n).astype(np.int64)
    x = omoe.as_f32(wl.x)
    wg = omoe.as_f32(wl.gate_w)
    bias = None if wl.bias is None else wl.bias.numpy()
    ids, _ = omoe.topk_route(omoe.router_logits(x[tokens], wg, bias), s.K)
    experts = [int(e) for e in np.unique(ids)]
    bits = lambda t: t.contiguous().view(__import__("torch").int16).numpy().view(np.uint16)
    ctx = mp.get_context("spawn")
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"
    with tempfile.TemporaryDirectory(prefix="moe_oracle_") as path:
        np.save(os.path.join(path, "x.npy"), x)
        np.save(os.path.join(path, "wg.npy"), wg)
        if bias is not None:
            np.save(os.path.join(path, "bias.npy"), bias)
        E, H, I = s.E, s.H, s.I
        mm = {}
        for name, (N, Kd) in (("w13", (2 * I, H)), ("w2", (H, I))):
            mm[name] = (np.lib.format.open_memmap(os.path.join(path, f"{name}_codes.npy"), "w+", np.uint8, (E, N, Kd)),
                        np.lib.format.open_memmap(os.path.join(path, f"{name}_sf.npy"), "w+", np.uint8,
                                                  (E, N, Kd // 16)),
                        np.ones(E, np.float32))
        with ctx.Pool(max(1, min(16, len(affinity())))) as pool:
            jobs = [(bits(wl.w13[e]), bits(wl.w2[e])) for e in experts]
            for e, (q13, q2) in zip(experts, pool.map(_oracle_quantize, jobs)):
                for name, q in (("w13", q13), ("w2", q2)):
                    mm[name][0][e], mm[name][1][e], mm[name][2][e] = q
        for name in mm:
            mm[name][0].flush()
            mm[name][1].flush()
            np.save(os.path.join(path, f"{name}_gs.npy"), mm[name][2])
        del mm
        if shared is not None:
            for name, w in (("s13", shared[0]), ("s2", shared[1])):
                qs = omoe.quantize_weights(omoe.as_f32(w)[None])
                np.save(os.path.join(path, f"{name}_codes.npy"), qs.codes)
                np.save(os.path.join(path, f"{name}_sf.npy"), qs.sf)
                np.save(os.path.join(path, f"{name}_gs.npy"), qs.gs)
        barrier = ctx.Barrier(procs)
        queue = ctx.Queue()
        chunks = np.array_split(tokens, procs)
        ps = [ctx.Process(target=_oracle_proc, args=(path, c, steps, warmup, s.K, shared_average, barrier, queue))
              for c in chunks]
        for p_ in ps:
            p_.start()
        res = [queue.get() for _ in ps]
        for p_ in ps:
            p_.join()
    value = sum(nt / statistics.mean(t) for nt, t in res)
    mean_step = statistics.mean(statistics.mean(t) for _, t in res)
    cpus = affinity()
    return dict(value=value, unit="tokens/s", cores=procs, kind="oracle",
                sample=f"{n} of the workload's {wl.T} tokens per step over {procs} single-threaded processes "
                       f"({per_proc} each; {len(experts)} experts), {steps} timed steps after {warmup} warm-up, "
                       f"forward only (weight conversion untimed)",
                nproc=os.cpu_count(), affinity=_ranges(cpus), seconds_per_step=mean_step)


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
    """(hbm GB/s, dense bf16 TFLOP/s burst, kind): the driver's measured peaks,
    else the stated fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# The sources that fix a GEMM launch's DRAM traffic: the kernel, its shared
# device helpers and argument block, and the host code that sizes its grid.
GEMM_SOURCES = ("common.cuh", "kernels.h", "kernels_gemm.cu", "moe_host.cu")


def _code_only(text):
    """C++ source with its comments removed and whitespace collapsed, so that
    a comment edit does not count as a change of the kernel.  (The GEMM
    sources hold no string literal with a comment marker in it.)"""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "nvfp4_token_quantized_gb300", "csrc")
    for f in GEMM_SOURCES:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode() + _code_only(fh.read()).encode())
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


def stage_flops(s, T):
    """Algorithmic FLOPs of the two expert GEMMs (2 per multiply-add)."""
    R = T * s.K
    return {"gemm_w13": 2 * R * s.H * 2 * s.I, "gemm_w2": 2 * R * s.I * s.H}


def layer_alg_bytes(s, T, touched, shared_inter=0):
    # x in, out, router weight, and the NVFP4 weights of the experts that got
    # rows (and of the shared expert)
    return (2 * T * s.H + 2 * T * s.H + 2 * s.H * s.E
            + (touched * 3 * s.I + 3 * shared_inter) * s.H * NVFP4_BYTES_PER_ELT)


def layer_flops(s, T, shared_inter=0):
    return 6 * T * s.K * s.H * s.I + 6 * T * s.H * shared_inter


# --------------------------------------------------------------------------
# Our implementation
# --------------------------------------------------------------------------

def workload_config(s, T, world, shared_inter=0, shared_average=False, accurate_sigmoid=False,
                    how="CUDA-graph replay"):
    extra = {}
    shared_desc = ""
    if shared_inter:
        combine = "average" if shared_average else "sum"
        extra = {"shared_inter": shared_inter, "shared_combine": combine}
        shared_desc = f" + shared expert Is={shared_inter} ({combine}, second stream)"
    if accurate_sigmoid:
        extra["sigmoid"] = "1/(1+expf(-g))"
    return {"workload": f"{s.name}: T={T} H={s.H} E={s.E} top-{s.K} I={s.I} on an instance for "
                        f"{s.max_num_tokens} tokens{shared_desc}, {how}",
            "T": T, "H": s.H, "E": s.E, "top_k": s.K, "I": s.I, "max_num_tokens": s.max_num_tokens,
            "deterministic": s.deterministic, "routing": "Zipf(1.2) expert bias" if s.zipf_bias else "random gate",
            **extra,
            "finalize": ("ordered: bf16 (token, slot) rows summed in slot order" if ordered_finalize(s, T)
                         else "fp32 atomic in the w2 epilogue"),
            "l2": "flushed before every step outside the timed events: a 256 MB write, then a 256 MB read of "
                  "another buffer so the flush's own dirty lines are written back before timing (the weights, "
                  "over 300 MB, also exceed L2)",
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


def roofline_summary(s, T, touched, step_ms, stage_ms, shared_inter, config_name):
    """Dominant kernel against HBM, the expert GEMMs against the FP4 tensor
    peak, and the whole layer against max(FLOP / FP4 peak, bytes / HBM)."""
    hbm, bf16, kind = measured_peaks()
    fp4 = bf16 * FP4_OVER_BF16
    dom = max(stage_ms, key=stage_ms.get)
    alg = stage_alg_bytes(s, T, touched)
    achieved = alg[dom] / (stage_ms[dom] / 1e3) / 1e9
    fl = stage_flops(s, T)
    g13 = fl["gemm_w13"] / (stage_ms["gemm_w13"] / 1e3) / 1e12
    gboth = (fl["gemm_w13"] + fl["gemm_w2"]) / ((stage_ms["gemm_w13"] + stage_ms["gemm_w2"]) / 1e3) / 1e12
    lb = layer_alg_bytes(s, T, touched, shared_inter)
    lf = layer_flops(s, T, shared_inter)
    t_hbm = lb / (hbm * 1e9) * 1e3
    t_fp4 = lf / (fp4 * 1e12) * 1e3
    return {
        "roofline": {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "peak_kind": f"{kind} hbm_gbs",
                     "alg_bytes_per_launch": alg[dom], "launch_ms": stage_ms[dom],
                     "traffic": dram_traffic(dom, config_name)},
        "roofline_fp4": {"kernel": "gemm_w13", "bound": "tensor", "achieved": g13, "peak": fp4, "unit": "TFLOP/s",
                         "frac": g13 / fp4, "flops_per_launch": fl["gemm_w13"], "launch_ms": stage_ms["gemm_w13"],
                         "both_gemms_frac": gboth / fp4,
                         "peak_kind": f"{kind} bf16_tflops x {FP4_OVER_BF16:g} (nominal dense FP4 / bf16 = "
                                      f"13.5 / 2.25 PFLOP/s)"},
        "layer_roofline": {"bound": "hbm" if t_hbm >= t_fp4 else "tensor", "alg_bytes": lb, "flops": lf,
                           "roofline_ms": max(t_hbm, t_fp4), "hbm_ms": t_hbm, "fp4_ms": t_fp4,
                           "frac": max(t_hbm, t_fp4) / step_ms, "achieved_gbs": lb / (step_ms / 1e3) / 1e9,
                           "achieved_tflops": lf / (step_ms / 1e3) / 1e12, "touched_experts": touched},
    }


def run_config(args, name, T, rank, world, local_rank):
    """Time one workload on this rank's GPU.  Returns the per-rank result
    (every rank) with the timings already maxed over ranks."""
    import torch

    from nvfp4_token_quantized_gb300 import MoE

    import synthetic

    dev = torch.device("cuda", local_rank)
    wl = workload(name, T)
    s = wl.shape
    T = wl.T
    Is = args.shared_inter
    layer = MoE(s.H, s.I, s.E, s.K, s.max_num_tokens, device=local_rank, deterministic=s.deterministic,
                shared_inter=Is, shared_average=args.shared_average, accurate_sigmoid=args.accurate_sigmoid)
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

    # Two CUDA graphs of one forward: the timed graph has no instrumentation;
    # the second records an event at every kernel boundary for the per-stage
    # breakdown and the roofline of the dominant kernel (its boundary events
    # serialise the kernels they separate).
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

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with torch.cuda.stream(stream):
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
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            flush_l2(i)
            starts[i].record(stream)
            graph.replay()
            ends[i].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]

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
    layer.close()

    med = statistics.median(step_ms)
    med, mean_ms, total_ms, e2e_med = max_over_ranks(
        [med, statistics.mean(step_ms), sum(step_ms), statistics.median(e2e_s)], world)
    stage_med = {k: statistics.median(v) for k, v in stages.items() if v}
    res = {
        "metric": METRIC,
        "value": replica_throughput(T, world, med),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": med,
        "ms_per_step_mean": mean_ms,
        "timed_ms_total": total_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "nvfp4 (e2m1 x e2m1 with e4m3 block scales, fp32 accumulate)",
        "data": "synthetic (seeded bf16 N(0,1) activations, N(0,0.02) router/expert weights)",
        "config": workload_config(s, T, world, Is, args.shared_average, args.accurate_sigmoid),
    }
    res.update(roofline_summary(s, T, touched, med, stage_med, Is, name))
    res.update({
        "stages_ms": stage_med,
        "stages_note": "median per-kernel times from an instrumented replay whose boundary events serialise the "
                       "kernels",
        "e2e": {"value": T * world / e2e_med, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_med * 1e3,
                "path": "moe_forward_host (pinned host buffers, eager launches, median step)"},
        "gpu_launches": kernels_per_forward(s, T, Is) * args.steps,
        "clocks": clk,
    })
    return res, wl


def cpu_baseline_for(args, wl):
    """The oracle on the host cores for the same workload: all cores of the
    affinity mask (at most 16 processes), plus one process alone."""
    per = args.cpu_sample or 4
    procs = args.cpu_procs or max(1, min(16, len(affinity())))
    shared = None
    if args.shared_inter:
        import synthetic

        shared = synthetic.make_shared_weights(wl.shape, args.shared_inter)
    allc = run_oracle(wl, steps=3, warmup=1, per_proc=per, procs=procs, shared=shared,
                      shared_average=args.shared_average)
    one = run_oracle(wl, steps=3, warmup=1, per_proc=per, procs=1, shared=shared,
                     shared_average=args.shared_average)
    out = {k: allc[k] for k in ("value", "unit", "cores", "kind", "sample", "nproc", "affinity")}
    out["single_thread"] = {k: one[k] for k in ("value", "unit", "cores", "sample")}
    return out


def run_ours(args, rank, world, local_rank):
    import torch

    from nvfp4_token_quantized_gb300 import build

    build()
    torch.cuda.set_device(local_rank)
    if args.config == "all":
        names = list(PER_CONFIG) + [HEADLINE]
    else:
        names = [args.config]
    results, workloads = {}, {}
    for name in names:
        T = args.tokens if args.config != "all" else None
        results[name], workloads[name] = run_config(args, name, T, rank, world, local_rank)
    if rank != 0:
        return None
    head_name = HEADLINE if args.config == "all" else args.config
    res = results[head_name]
    if args.config == "all":
        keep = ("value", "unit", "ms_per_step", "ms_per_step_mean", "config", "roofline", "roofline_fp4",
                "layer_roofline", "stages_ms", "e2e", "gpu_launches", "clocks")
        res["per_config"] = {n: {k: results[n][k] for k in keep} for n in PER_CONFIG}
    if world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline_for(args, workloads[head_name])
    return res


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        name = HEADLINE if args.config == "all" else args.config
        wl = workload(name, args.tokens if args.config != "all" else None)
        procs = args.cpu_procs or max(1, min(16, len(affinity())))
        shared = None
        if args.shared_inter:
            import synthetic

            shared = synthetic.make_shared_weights(wl.shape, args.shared_inter)
        r = run_oracle(wl, steps=max(1, args.steps), warmup=args.warmup, per_proc=args.cpu_sample or 1,
                       procs=procs, shared=shared, shared_average=args.shared_average)
        line = {"impl": "reference", "metric": METRIC, "value": r["value"], "unit": "tokens/s", "n_gpus": 1,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["seconds_per_step"] * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
                "data": "synthetic", "config": workload_config(wl.shape, wl.T, 1, args.shared_inter,
                                                          args.shared_average, how="the CPU oracle"),
                "cpu_baseline": {k: r[k] for k in ("value", "unit", "cores", "kind", "sample", "nproc", "affinity")},
                "e2e": {"value": r["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("gloo", rank=rank, world_size=world)
    res = run_ours(args, rank, world, local_rank)
    if res is not None:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
