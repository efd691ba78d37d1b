#!/usr/bin/env python
"""Throughput of the sparse MoE layer forward pass on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one whole layer forward (router, top-k, capacity dispatch + gather,
expert GEMMs, combine) over one batch of seeded synthetic tokens already
resident in HBM, issued through the C ABI (moe_forward_timed).  The timed
steps are replayed as CUDA graphs (--eager: launched from the host); L2 is
flushed (256 MiB write) between timed steps, outside the measured events.
Prints one JSON line.  Besides the layer, the line carries `routing_stats`:
the time of one moe_routing_stats call over the same batch (routing
diagnostics and auxiliary load-balancing loss; L2 flushed before each call)
and the values it returned.

--impl reference times the fp64 CPU oracle instead (the reference arm of this
benchmark), on the host cores, each step a bounded sub-batch of the workload.
For N > 1 (torchrun) every rank runs an independent replica of the layer on
its own GPU and batch: the path has no exchange step, so there is no
collective on the data path; ranks only meet at the barriers around the
timed region and in the max-over-ranks of the elapsed time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer fwd tokens/s on 1 B300; TFLOP/s or HBM GB/s as % of roofline"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "bf16_t4096"
FLUSH_BYTES = 256 << 20

# DRAM traffic of the dominant kernel per launch, from an ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), keyed by workload and by the
# hash of the kernel sources it was taken on; a changed kernel reports null.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
GEMM_SOURCES = ["sparse_mixture_experts_51_b300/csrc/gemm_tc.cu", "sparse_mixture_experts_51_b300/csrc/common.cuh"]


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU-baseline sample budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true", help="launch every kernel from the host (no CUDA graph)")
    return ap.parse_args(argv)


# ---------------------------------------------------------------- helpers

def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def step_quantiles(step_ms):
    """Median and 95th percentile of the per-step device times (ms, this rank)."""
    v = sorted(step_ms)
    if not v:
        return None
    return {"p50": statistics.median(v), "p95": v[min(len(v) - 1, math.ceil(0.95 * len(v)) - 1)]}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), source="measured")
    return dict(hbm_gbs=6400.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0, source="fallback")


def gemm1_work(w, counts):
    """Algorithmic flops and DRAM bytes of the first expert GEMM (dominant kernel)
    for the kept rows: flops 2*d*F per row (x2 for SwiGLU's gate and up),
    bytes = weights of every expert with a kept row + grouped rows read + hidden written."""
    from sparse_mixture_experts_51_b300 import workloads as W
    R = int(sum(counts))
    active = sum(1 for c in counts if c > 0)
    b = 2 if w.dtype_name == "bf16" else 4
    mats = 2 if w.act == W.ACT_SWIGLU else 1
    flops = float(R) * 2.0 * w.d * w.F * mats
    nbytes = float(active) * mats * w.F * w.d * b + float(R) * w.d * b + float(R) * w.F * b
    return flops, nbytes


class ClockSampler:
    """Samples the SM clock and the clock-event (throttle) reasons while the
    timed region runs: through NVML when it loads, else by polling nvidia-smi."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
               0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}
    SMI_FIELDS = ("clocks.sm,clocks.max.sm,utilization.gpu,clocks_event_reasons.gpu_idle,"
                  "clocks_event_reasons.sw_power_cap,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown")

    def __init__(self, index: int, period_s: float = 0.01):
        self.index = index
        self.samples = []  # (mhz, reason bits)
        self.max_mhz = None
        self.mode = None
        self.err = ""
        self._stop = threading.Event()
        self.period = period_s
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nv = pynvml
            self.h = pynvml.nvmlDeviceGetHandleByIndex(index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.mode = "nvml"
        except Exception as e:
            self.err = repr(e)
            import shutil
            if shutil.which("nvidia-smi"):
                self.mode = "nvidia-smi"

    def _run_nvml(self):
        nv = self.nv
        fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            try:
                self.samples.append((nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM), int(fn(self.h))))
            except Exception:
                pass
            time.sleep(self.period)

    def wait_started(self, timeout_s: float = 3.0):
        """Returns once the first clock sample is in (or after timeout_s)."""
        t0 = time.time()
        if self.mode == "nvml":
            while not self.samples and time.time() - t0 < timeout_s:
                time.sleep(0.005)
        elif self.mode == "nvidia-smi":
            # nvidia-smi prints its first sample right after it starts
            while time.time() - t0 < min(timeout_s, 1.0):
                time.sleep(0.05)

    def __enter__(self):
        if self.mode == "nvml":
            self.t = threading.Thread(target=self._run_nvml, daemon=True)
            self.t.start()
        elif self.mode == "nvidia-smi":
            import subprocess
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.SMI_FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        return self

    def __exit__(self, *a):
        if self.mode == "nvml":
            self._stop.set()
            self.t.join()
        elif self.mode == "nvidia-smi":
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            bits_of = [0x1, 0x4, 0x8, 0x40, 0x20]
            for line in out.splitlines():
                f = [v.strip() for v in line.split(",")]
                if len(f) < 8:
                    continue
                try:
                    mhz, mx = float(f[0]), float(f[1])
                except ValueError:
                    continue
                bits = 0
                for b, v in zip(bits_of, f[3:8]):
                    if v.lower().startswith("active"):
                        bits |= b
                self.max_mhz = mx
                self.samples.append((mhz, bits))

    def summary(self):
        if self.mode is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "no clock source: " + self.err}
        busy = [s for s in self.samples if not (s[1] & 0x1)] or self.samples
        mhz = [s[0] for s in busy]
        bits = 0
        for s in busy:
            bits |= s[1]
        reasons = [name for bit, name in self.REASONS.items() if bits & bit and bit != 0x1]
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(busy), "source": self.mode}


_ORACLE_CACHE = {}


def cpu_oracle_run(w, budget_s: float):
    """Time the fp64 oracle, as it stands, on a sub-batch of the workload (the
    same layer with its first T_s tokens as their own batch) for about
    budget_s seconds.  Returns (tokens/s, sample description, threads, seconds)."""
    from oracle import moe_oracle as O
    from sparse_mixture_experts_51_b300 import workloads as W

    class F64:
        def __init__(self, t):
            self.t = t
            self.cache = {}

        def __getitem__(self, e):
            if e not in self.cache:
                self.cache[e] = W.as_f64_numpy(self.t[e])
            return self.cache[e]

    # sub-batch size from the algorithmic work per token (fp64 BLAS ~1e11 flop/s)
    per_tok = 2.0 * w.d * (3 if w.act == W.ACT_SWIGLU else 2) * (w.F * w.k + w.n_shared * w.F_shared) + 2.0 * w.d * w.E
    T_s = int(max(16, min(w.T, budget_s * 1e11 / per_tok / 2)))
    key = (w.name, T_s)
    if key not in _ORACLE_CACHE:
        inp = W.make_inputs(w.scaled(T_s))
        f = W.as_f64_numpy
        _ORACLE_CACHE[key] = (f(inp["x"]), f(inp["W_g"]), F64(inp["W1"]), F64(inp["W2"]), dict(
            W3=None if inp["W3"] is None else F64(inp["W3"]), b1=None if inp["b1"] is None else F64(inp["b1"]),
            b2=None if inp["b2"] is None else F64(inp["b2"]), b_g=f(inp["b_g"]), W_noise=f(inp["W_noise"]),
            eps=f(inp["eps"]), capacity_factor=w.capacity_factor,
            shared=None if inp["W1s"] is None else dict(
                W1s=f(inp["W1s"]), W2s=f(inp["W2s"]), W3s=f(inp["W3s"]), b1s=f(inp["b1s"]), b2s=f(inp["b2s"]))))
    x, Wg, W1, W2, args = _ORACLE_CACHE[key]
    runs, tokens, t0 = 0, 0, time.perf_counter()
    while True:
        if w.routing == "expert":
            O.forward_expert_choice(x, Wg, w.act, W1, W2, k=w.k, **args)
        else:
            O.forward(x, Wg, w.k, w.act, W1, W2, **args)
        runs += 1
        tokens += T_s
        el = time.perf_counter() - t0
        if el >= budget_s or runs >= 1000:
            break
    cores = os.cpu_count()
    sample = (f"{runs} oracle forward(s) of a {T_s}-token sub-batch of {w.name} (its own capacity "
              f"ceil({w.capacity_factor}*{T_s}*{w.k}/{w.E})), fp64 NumPy, BLAS on all host threads")
    return tokens / el, sample, cores, el


# ---------------------------------------------------------------- ranks
# bench.py under torchrun runs one independent replica of the layer per GPU:
# the path has no exchange step.  These helpers hold the host-side logic of
# that mode (tested with gloo ranks on the CPU).

def replica_workload(w, rank: int, world: int):
    """Rank r's replica: the same layer with its own token batch (seed + 1000 r)."""
    return w.with_(seed=w.seed + 1000 * rank) if world > 1 else w


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest value over all ranks (the slowest rank sets the job's time)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank_step: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank_step * steps * world / (max_ms / 1e3)


# ---------------------------------------------------------------- arms

def run_reference(a):
    """Reference arm: the fp64 CPU oracle, timed on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from sparse_mixture_experts_51_b300 import workloads as W
    w = W.WORKLOADS[a.workload]
    per_step = max(0.5, min(10.0, 150.0 / max(1, a.steps + a.warmup)))
    for i in range(a.warmup):
        cpu_oracle_run(w, per_step * 0.2)
    vals, total_t, total_tok = [], 0.0, 0.0
    sample = ""
    cores = os.cpu_count()
    for i in range(a.steps):
        v, sample, cores, el = cpu_oracle_run(w, per_step)
        vals.append(v)
        total_t += el
        total_tok += v * el
    value = total_tok / total_t
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": a.gpus, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": 1e3 * total_t / a.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def workload_config(w):
    from sparse_mixture_experts_51_b300 import workloads as W
    return {"workload": w.name, "T": w.T, "d": w.d, "E": w.E, "k": w.k, "d_ff": w.F,
            "act": "swiglu" if w.act == W.ACT_SWIGLU else "gelu", "capacity_factor": w.capacity_factor,
            "noisy_gating": w.noisy, "dtype": w.dtype_name, "seed": w.seed,
            **({"shared_experts": w.n_shared, "d_ff_shared_each": w.F_shared} if w.n_shared else {}),
            **({"routing": "expert_choice"} if w.routing == "expert" else {}),
            "l2": "flushed between timed steps (256 MiB write, outside the timed events)"}


def run_ours(a):
    import ctypes

    import torch
    import torch.distributed as dist

    from sparse_mixture_experts_51_b300 import _lib, api
    from sparse_mixture_experts_51_b300 import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    lib = _lib.load()

    w = replica_workload(W.WORKLOADS[a.workload], rank, world)
    inp = W.make_inputs(w)
    g = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    act = "swiglu" if w.act == W.ACT_SWIGLU else "gelu"
    C = api.capacity(w.T, w.k, w.E, w.capacity_factor)
    sw = W.shared_wide(g)
    Fsh = 0 if sw["W1s"] is None else sw["W1s"].shape[0]
    shape = api.shape_of(w.T, w.d, w.E, w.k, w.F, w.dtype, act, d_ff_shared=Fsh, routing=w.routing)
    shared_w = None
    if Fsh:
        b2s = None if sw["b2s_rows"] is None else sw["b2s_rows"].sum(dim=0).contiguous()
        shared_t = dict(W1s=sw["W1s"], W2s=sw["W2s"], W3s=sw["W3s"], b1s=sw["b1s"], b2s=b2s)
        shared_w = api.shared_weights(**shared_t)
    shared_arg = ctypes.addressof(shared_w) if shared_w is not None else None
    ws = api.new_workspace(shape, C, dev)
    out = torch.empty(w.T, w.d, dtype=w.dtype, device=dev)
    counts = torch.empty(w.E, dtype=torch.int32, device=dev)
    dropped = torch.empty(1, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    P = api._ptr

    def fwd_args():
        # the stream current at the call (the capture stream while a graph is recorded)
        sptr = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
        return [ctypes.byref(shape), float(w.capacity_factor), -1, P(g["x"]), P(g["W_g"]), P(g["b_g"]),
                P(g["W_noise"]), P(g["eps"]), P(g["W1"]), P(g["W3"]), P(g["W2"]), P(g["b1"]), P(g["b2"]), shared_arg,
                P(out), None, None, None, None, P(counts), None, P(dropped), None, None, P(ws), ws.numel(), sptr]

    # the timed steps run as CUDA graphs of up to GRAPH_STEPS steps each (every
    # step the same C-ABI call, moe_forward_timed, its launches replayed
    # without host gaps); the L2 flush between steps lies outside each
    # step's events, and the events of a graph are read after each replay
    GRAPH_STEPS = 250
    G = min(a.steps, GRAPH_STEPS)
    stage_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(G)]

    # events before the router, around expert GEMM 1 (the roofline kernel) and
    # after the combine; none inside the router -> dispatch -> gather and
    # GEMM 2 -> combine chains, whose kernels overlap their neighbours'
    # tails through programmatic dependent launch
    def step_timed(i):
        evs = stage_ev[i]
        arr = (ctypes.c_void_p * 6)(ctypes.c_void_p(evs[0].cuda_event), None, ctypes.c_void_p(evs[2].cuda_event),
                                    ctypes.c_void_p(evs[3].cuda_event), None, ctypes.c_void_p(evs[5].cuda_event))
        _lib.check(lib.moe_forward_timed(*fwd_args(), arr), "moe_forward_timed")

    # make sure every event exists on the device before its handle is used
    for evs in stage_ev:
        for e in evs:
            e.record(stream)
    torch.cuda.synchronize()

    for _ in range(a.warmup):
        _lib.check(lib.moe_forward(*fwd_args()), "moe_forward")
        flush.zero_()
    torch.cuda.synchronize()
    assert api.get_device_error(ws) == 0
    # kernels one step enqueues (the library counts its own launches; a graph
    # replays exactly what one captured call enqueued)
    n0 = lib.moe_kernel_launches()
    _lib.check(lib.moe_forward(*fwd_args()), "moe_forward")
    kernels_per_step = int(lib.moe_kernel_launches() - n0)
    torch.cuda.synchronize()

    graphs = {}

    def graph_of(n):
        if n not in graphs:
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr):
                for i in range(n):
                    flush.zero_()
                    step_timed(i)
            torch.cuda.synchronize()
            graphs[n] = gr
        return graphs[n]

    chunks = [G] * (a.steps // G) + ([a.steps % G] if a.steps % G else [])
    if not a.eager:
        for n in set(chunks):
            graph_of(n)

    step_ms, stage_ms = [], [[] for _ in range(3)]
    SPANS = [(0, 2), (2, 3), (3, 5)]  # router+dispatch+gather, expert GEMM 1, expert GEMM 2+combine
    sampler = ClockSampler(local)
    with sampler:
        sampler.wait_started()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        for n in chunks:
            if a.eager:
                for i in range(n):
                    flush.zero_()
                    step_timed(i)
            else:
                graphs[n].replay()
            torch.cuda.synchronize()
            step_ms += [evs[0].elapsed_time(evs[5]) for evs in stage_ev[:n]]
            for j, (u, v) in enumerate(SPANS):
                stage_ms[j] += [evs[u].elapsed_time(evs[v]) for evs in stage_ev[:n]]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
    err = api.get_device_error(ws)
    if err != 0:
        raise RuntimeError(f"device-side error {err} during the timed region")

    total_ms = max_over_ranks(sum(step_ms), world, dev)
    value = job_throughput(w.T, a.steps, world, total_ms)

    # ---------------- roofline of the dominant kernel (first expert GEMM)
    cnt = counts.cpu().tolist()
    flops, nbytes = gemm1_work(w, cnt)
    g1_ms = statistics.mean(stage_ms[1])
    peaks = load_peaks()
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    traffic = None
    if os.path.exists(TRAFFIC_FILE):
        with open(TRAFFIC_FILE) as fh:
            rec = json.load(fh).get(w.name)
        if rec and rec.get("kernel_hash") == kernel_hash():
            traffic = rec.get("dram_bytes_per_launch")
    if flops / nbytes >= ridge:
        achieved = flops / (g1_ms / 1e3) / 1e12
        roof = {"kernel": "grouped_gemm_kernel (expert GEMM 1, fused activation)", "bound": "tensor",
                "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"], "peak_source": peaks["source"] + " bf16 burst",
                "algorithmic_flops": flops, "ms_per_launch": g1_ms, "traffic": traffic}
    else:
        achieved = nbytes / (g1_ms / 1e3) / 1e9
        roof = {"kernel": "grouped_gemm_kernel (expert GEMM 1, fused activation)", "bound": "hbm",
                "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "peak_source": peaks["source"] + " copy bandwidth",
                "algorithmic_bytes": nbytes, "ms_per_launch": g1_ms, "traffic": traffic}

    # ---------------- end to end through the public API with host buffers.
    # Every step copies its tokens (and noise) from pinned host memory, runs
    # the layer (MoELayer, the public call) and reads the output back to
    # pinned host memory.  Like a serving loop the steps are pipelined on
    # three streams with two device buffer sets: the input copy of step i+1
    # and the output copy of step i-1 overlap the layer of step i.  The timed
    # region spans the first input copy to the last output copy; no L2 flush
    # (every step's inputs arrive from the host, and the expert weights are
    # read from HBM each step).
    layer = api.MoELayer(g["W_g"], g["W1"], g["W2"], w.k, act, W3=g["W3"], b_g=g["b_g"], W_noise=g["W_noise"],
                         b1=g["b1"], b2=g["b2"], capacity_factor=w.capacity_factor, keep_routing=False,
                         routing=w.routing, **(shared_t if Fsh else {}))
    x_host = inp["x"].pin_memory()
    eps_host = inp["eps"].pin_memory() if inp["eps"] is not None else None
    out_host = [torch.empty(w.T, w.d, dtype=w.dtype).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(g["x"]) for _ in range(2)]
    eps_dev = [torch.empty_like(g["eps"]) if g["eps"] is not None else None for _ in range(2)]
    out_dev = [torch.empty_like(out) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_run(n):
        """n pipelined steps; returns the elapsed ms from the first input copy to the last output copy."""
        ev = lambda: torch.cuda.Event(enable_timing=False)
        in_ready, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        s_in.wait_event(t0)
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(comp_done[b])  # the layer of step i-2 has read this buffer
                x_dev[b].copy_(x_host, non_blocking=True)
                if eps_host is not None:
                    eps_dev[b].copy_(eps_host, non_blocking=True)
                in_ready[b].record(s_in)
            stream.wait_event(in_ready[b])
            if i >= 2:
                stream.wait_event(out_done[b])  # the output of step i-2 has left this buffer
            layer(x_dev[b], eps=eps_dev[b], out=out_dev[b], stream=stream)
            comp_done[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[b])
                out_host[b].copy_(out_dev[b], non_blocking=True)
                out_done[b].record(s_out)
        stream.wait_event(out_done[(n - 1) % 2])
        if n >= 2:
            stream.wait_event(out_done[n % 2])
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    e2e_run(max(2, a.warmup))
    n_e2e = max(2, a.steps)
    e2e_ms = max_over_ranks(e2e_run(n_e2e), world, dev)
    # the layer run through the public call gives the device-timed output, bit for bit
    if not torch.equal(out_host[(n_e2e - 1) % 2], out.cpu()):
        raise RuntimeError("end-to-end output differs from the timed layer's output")
    h2d = x_host.numel() * x_host.element_size() + (eps_host.numel() * 4 if eps_host is not None else 0)
    d2h = out_host[0].numel() * out_host[0].element_size()
    e2e = {"value": job_throughput(w.T, n_e2e, world, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "pipelined": "input copy of step i+1 and output copy of step i-1 overlap "
                                                   "the layer of step i (two buffer sets, three streams)"}

    # ---------------- routing diagnostics + aux loss of the same batch (moe_routing_stats,
    # a separate call after the layer; token-choice routing only, it needs a top-k table)
    routing_stats = None
    n_st = 50
    sptr = ctypes.c_void_p(stream.cuda_stream)
    if w.routing == "token":
        logits = torch.empty(w.T, w.E, dtype=torch.float32, device=dev)
        idx_t = torch.empty(w.T, w.k, dtype=torch.int32, device=dev)
        fa = fwd_args()
        fa[16], fa[23] = P(idx_t), P(logits)
        _lib.check(lib.moe_forward(*fa), "moe_forward")
        st_out = [torch.empty(n, dtype=torch.float64, device=dev) for n in (w.E, w.E, len(api.STATS_SUMMARY))]
        sptr = ctypes.c_void_p(stream.cuda_stream)

        def stats_call():
            _lib.check(lib.moe_routing_stats(ctypes.byref(shape), P(logits), P(idx_t), P(counts), P(dropped),
                                             P(st_out[0]), P(st_out[1]), P(st_out[2]), P(ws), ws.numel(), sptr),
                       "moe_routing_stats")

        for _ in range(3):
            stats_call()
        # the call follows the layer, whose router has just written the logits,
        # so its inputs are L2-resident: time a CUDA graph of n_st back-to-back
        # calls (no host gaps between launches), after a warm-up replay
        torch.cuda.synchronize()
        gst = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gst):
            sptr = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
            for _ in range(n_st):
                stats_call()
        sptr = ctypes.c_void_p(stream.cuda_stream)
        gst.replay()
        sev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        sev[0].record(stream)
        gst.replay()
        sev[1].record(stream)
        torch.cuda.synchronize()
        if api.get_device_error(ws) != 0:
            raise RuntimeError("device-side error in moe_routing_stats")
        st_ms = sev[0].elapsed_time(sev[1]) / n_st
        st_bytes = w.T * w.E * 4 + w.T * w.k * 4  # logits + top-k table, read once
        summ = dict(zip(api.STATS_SUMMARY, st_out[2].tolist()))
        routing_stats = {"us_per_call": st_ms * 1e3, "timing": f"CUDA graph of {n_st} back-to-back calls, inputs L2-resident",
                         "algorithmic_bytes": st_bytes,
                         "achieved_gbs": st_bytes / (st_ms / 1e3) / 1e9,
                         "frac_hbm": st_bytes / (st_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                         "aux_loss": summ["aux_loss"], "entropy": summ["entropy"], "load_cv": summ["load_cv"],
                         "overflow": summ["overflow"]}

    # ---------------- the shared experts alone (moe_shared_ffn: two dense GEMMs over
    # every token), kernel time with L2 flushed before each call
    shared_ffn = None
    if Fsh:
        y_sh = torch.empty(w.T, w.d, dtype=torch.float32, device=dev)

        def shared_call():
            _lib.check(lib.moe_shared_ffn(ctypes.byref(shape), P(g["x"]), shared_arg, P(y_sh), P(ws), ws.numel(),
                                          sptr), "moe_shared_ffn")

        for _ in range(3):
            shared_call()
        hev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_st)]
        for i in range(n_st):
            flush.zero_()
            hev[i][0].record(stream)
            shared_call()
            hev[i][1].record(stream)
        torch.cuda.synchronize()
        if api.get_device_error(ws) != 0:
            raise RuntimeError("device-side error in moe_shared_ffn")
        sh_ms = statistics.mean(s_.elapsed_time(e_) for s_, e_ in hev)
        sh_flops = 2.0 * w.T * w.d * Fsh * ((2 if w.act == W.ACT_SWIGLU else 1) + 1)
        shared_ffn = {"us_per_call": sh_ms * 1e3, "algorithmic_flops": sh_flops,
                      "achieved_tflops": sh_flops / (sh_ms / 1e3) / 1e12,
                      "frac_bf16": sh_flops / (sh_ms / 1e3) / 1e12 / peaks["bf16_tflops"],
                      "peak_source": peaks["source"] + " bf16 burst", "launches_per_call": 2}

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return 0

    cpu = None
    if not a.no_cpu_baseline and world == 1:
        v, sample, cores, _ = cpu_oracle_run(w, a.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}

    cfg = workload_config(w)
    cfg.update({"C": C, "kept_rows": int(sum(cnt)), "dropped": int(dropped.item()),
                "parallelism": "replicas" if world > 1 else "single_gpu",
                "launch": "eager" if a.eager else f"CUDA graphs of up to {GRAPH_STEPS} timed steps (moe_forward_timed each)"})
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
            "ms_per_step": total_ms / a.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "step_ms_quantiles": step_quantiles(step_ms),
            "dtype": w.dtype_name, "data": "synthetic", "config": cfg,
            "stage_ms": {n: statistics.mean(v) for n, v in zip(
                [("shared_ffn_" if Fsh else "") + ("router_select_gather" if w.routing == "expert"
                                                     else "router_dispatch_gather"), "expert_gemm1",
                 "expert_gemm2_combine"], stage_ms)},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": kernels_per_step * a.steps,
            "clocks": sampler.summary(), "routing_stats": routing_stats}
    if shared_ffn is not None:
        line["shared_ffn"] = shared_ffn
    print(json.dumps(line))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main(argv=None):
    a = parse_args(argv)
    if a.impl == "reference":
        return run_reference(a)
    return run_ours(a)


if __name__ == "__main__":
    sys.exit(main())
