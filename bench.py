#!/usr/bin/env python
"""Throughput of the sparse MoE layer forward pass on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one whole layer forward (router, top-k, capacity dispatch + gather,
expert GEMMs, combine) over one batch of seeded synthetic tokens already
resident in HBM, issued through the C ABI (moe_forward_timed).  The timed
steps are replayed as CUDA graphs (--eager: launched from the host); L2 is
flushed (a 256 MiB write, then a 256 MiB read that writes the dirty lines
back) between timed steps, outside the measured events.

Prints one JSON line for the headline layer (--workload, by default the
Mixtral-shaped layer: T=16384, d=4096, E=8 top-2, SwiGLU d_ff=14336, no
drops).  At one GPU the line also carries `per_config`: the same measurement
(shorter) for each of the five layer configurations -- tiny fp32, bf16
T=4096, Mixtral-shaped, Switch-style top-1 with forced overflow, and the
decode-like T=128 layer -- each with its roofline (tensor TFLOP/s for the
compute-bound shapes, HBM GB/s for the weight-streaming ones), near-tie and
drop counts, end-to-end rate with host buffers, and the fp64 CPU oracle
timed on the host cores (all threads, and one thread for the small layers).
The line carries `routing_stats` too: one moe_routing_stats call over the
same batch (routing diagnostics and the auxiliary load-balancing loss).

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
DEFAULT_WORKLOAD = "mixtral_t16384"
FLUSH_BYTES = 256 << 20
# the five layer configurations, in their usual order (each gets a per_config entry)
PER_CONFIG = ["tiny_fp32", "bf16_t4096", "mixtral_t16384", "switch_top1", "decode_t128"]
PER_CONFIG_STEPS = 200
PER_CONFIG_E2E_STEPS = 40
# layers whose oracle is also timed on one host thread
SINGLE_THREAD_CPU = ("tiny_fp32", "bf16_t4096", "decode_t128")
# the ~8 TB/s HBM figure the weight-streaming layer's bandwidth target is quoted against
HBM_NOMINAL_GBS = 8000.0

# DRAM traffic of the dominant kernel per launch, from an ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), keyed by workload; each
# record lists the kernel sources it was taken on and their hash, and a
# record whose sources have changed since reports null.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU-baseline sample budget of the headline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="measure the headline layer only")
    ap.add_argument("--eager", action="store_true", help="launch every kernel from the host (no CUDA graph)")
    return ap.parse_args(argv)


# ---------------------------------------------------------------- helpers

def kernel_hash(sources) -> str:
    h = hashlib.sha256()
    for f in sources:
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


def cpu_model() -> str:
    """The host CPU's model name (as lscpu prints it)."""
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or "unknown"


def layer_work(w, counts):
    """Algorithmic work of one layer forward with the given kept counts per expert.

    flops: per kept row 2*d*F per expert matrix (W1, W3 for SwiGLU, W2);
    bytes: tokens read once, the weights of every expert with a kept row,
    the output written, the noise table when noisy, and the routing tables
    (idx, gates, slots: 12 bytes per assignment)."""
    from sparse_mixture_experts_51_b300 import workloads as W
    R = int(sum(counts))
    active = sum(1 for c in counts if c > 0)
    b = 2 if w.dtype_name == "bf16" else 4
    mats1 = 2 if w.act == W.ACT_SWIGLU else 1
    gemm1_flops = float(R) * 2.0 * w.d * w.F * mats1
    ffn_flops = gemm1_flops + float(R) * 2.0 * w.d * w.F
    weight_bytes = float(active) * (mats1 + 1) * w.F * w.d * b
    layer_bytes = (2.0 * w.T * w.d * b + weight_bytes + (w.T * w.E * 4.0 if w.noisy else 0.0) + 12.0 * w.T * w.k)
    gemm1_bytes = float(active) * mats1 * w.F * w.d * b + float(R) * w.d * b + float(R) * w.F * b
    return dict(kept_rows=R, active_experts=active, gemm1_flops=gemm1_flops, ffn_flops=ffn_flops,
                weight_bytes=weight_bytes, layer_bytes=layer_bytes, gemm1_bytes=gemm1_bytes)


def recorded_traffic(name):
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as fh:
        rec = json.load(fh).get(name)
    if rec and rec.get("sources") and rec.get("kernel_hash") == kernel_hash(rec["sources"]):
        return rec.get("dram_bytes_per_launch")
    return None


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


def _oracle_timed(w, budget_s: float, rate: float):
    """Time the fp64 oracle, as it stands, on a sub-batch of the workload (the
    same layer with its first T_s tokens as their own batch, T_s sized from
    the expected fp64 rate) for about budget_s seconds.
    Returns (tokens/s, runs, T_s, seconds)."""
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

    per_tok = 2.0 * w.d * (3 if w.act == W.ACT_SWIGLU else 2) * (w.F * w.k + w.n_shared * w.F_shared) + 2.0 * w.d * w.E
    T_s = int(max(16, min(w.T, budget_s * rate / per_tok / 2)))
    key = (w.name, w.seed, T_s)
    if key not in _ORACLE_CACHE:
        _ORACLE_CACHE.clear()  # one workload's widened weights at a time
        inp = W.make_inputs(w.scaled(T_s))
        f = W.as_f64_numpy
        _ORACLE_CACHE[key] = (f(inp["x"]), f(inp["W_g"]), F64(inp["W1"]), F64(inp["W2"]), dict(
            W3=None if inp["W3"] is None else F64(inp["W3"]), b1=None if inp["b1"] is None else F64(inp["b1"]),
            b2=None if inp["b2"] is None else F64(inp["b2"]), b_g=f(inp["b_g"]), W_noise=f(inp["W_noise"]),
            eps=f(inp["eps"]), capacity_factor=w.capacity_factor,
            shared=None if inp["W1s"] is None else dict(
                W1s=f(inp["W1s"]), W2s=f(inp["W2s"]), W3s=f(inp["W3s"]), b1s=f(inp["b1s"]), b2s=f(inp["b2s"]))))
    x, Wg, W1, W2, args = _ORACLE_CACHE[key]

    def run():
        if w.routing == "expert":
            O.forward_expert_choice(x, Wg, w.act, W1, W2, k=w.k, **args)
        else:
            O.forward(x, Wg, w.k, w.act, W1, W2, **args)

    run()  # widens the expert weights to fp64 once (not timed)
    runs, tokens, t0 = 0, 0, time.perf_counter()
    while True:
        run()
        runs += 1
        tokens += T_s
        el = time.perf_counter() - t0
        if el >= budget_s or runs >= 1000:
            break
    return tokens / el, runs, T_s, el


def _oracle_child(name: str, seed: int, budget_s: float, threads: int) -> None:
    """Entry point of the one-thread oracle sample (a fresh interpreter whose
    BLAS was loaded with its thread count set in the environment)."""
    from sparse_mixture_experts_51_b300 import workloads as W
    w = W.WORKLOADS[name].with_(seed=seed)
    print(json.dumps(_oracle_timed(w, budget_s, rate=5e9 * threads)))


def cpu_oracle_run(w, budget_s: float, threads=None):
    """The fp64 oracle on a bounded sub-batch of ``w`` for about budget_s
    seconds: in this process on all host threads, or (``threads`` given) in
    a child interpreter whose BLAS runs that many threads (BLAS libraries
    read their thread count when they load).
    Returns (tokens/s, sample description, threads used, seconds)."""
    if threads is None:
        v, runs, T_s, el = _oracle_timed(w, budget_s, rate=1e11)
        cores = os.cpu_count()
        how = "BLAS on all host threads"
    else:
        import subprocess
        env = dict(os.environ)
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS",
                    "VECLIB_MAXIMUM_THREADS", "NUMEXPR_NUM_THREADS"):
            env[var] = str(threads)
        code = (f"import sys; sys.path.insert(0, {ROOT!r}); import bench; "
                f"bench._oracle_child({w.name!r}, {int(w.seed)}, {float(budget_s)}, {int(threads)})")
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
        if r.returncode != 0:
            raise RuntimeError(f"one-thread oracle sample failed: {r.stderr[-2000:]}")
        v, runs, T_s, el = json.loads(r.stdout.strip().splitlines()[-1])
        cores = threads
        how = f"BLAS on {threads} thread(s) (a child process started with the BLAS thread variables set)"
    sample = (f"{runs} oracle forward(s) of a {T_s}-token sub-batch of {w.name} (its own capacity "
              f"ceil({w.capacity_factor}*{T_s}*{w.k}/{w.E})), fp64 NumPy, " + how)
    return v, sample, cores, el


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
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
                             "cpu_model": cpu_model()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def workload_config(w):
    """The workload as the JSON line's `config` (identical in both arms)."""
    from sparse_mixture_experts_51_b300 import workloads as W
    return {"workload": w.name, "T": w.T, "d": w.d, "E": w.E, "k": w.k, "d_ff": w.F,
            "act": "swiglu" if w.act == W.ACT_SWIGLU else "gelu", "capacity_factor": w.capacity_factor,
            "noisy_gating": w.noisy, "dtype": w.dtype_name, "seed": w.seed,
            **({"shared_experts": w.n_shared, "d_ff_shared_each": w.F_shared} if w.n_shared else {}),
            **({"routing": "expert_choice"} if w.routing == "expert" else {}),
            "l2": "flushed between timed steps (256 MiB write then 256 MiB read, outside the timed events)"}


class L2Flush:
    """Empties L2 between timed steps, outside their events: writes a buffer
    larger than L2, then reads a second one, so that the dirty lines the write
    leaves are written back here and not during the next step (whose weight
    stream would otherwise pay for about one L2 of write-backs)."""

    def __init__(self, dev, nbytes=FLUSH_BYTES):
        import torch
        self.w = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(nbytes // 8, dtype=torch.int64, device=dev)
        self.sink = torch.zeros((), dtype=torch.int64, device=dev)

    def __call__(self):
        import torch
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.sink)


class DeviceLayer:
    """One workload's layer resident on the GPU: inputs, weights, workspace and
    the argument list of moe_forward / moe_forward_timed."""

    def __init__(self, w, dev, lib, keep_host_tokens=True):
        import ctypes

        import torch

        from sparse_mixture_experts_51_b300 import api
        from sparse_mixture_experts_51_b300 import workloads as W

        self.w, self.dev, self.lib = w, dev, lib
        inp = W.make_inputs(w)
        self.x_host = inp["x"] if keep_host_tokens else None
        self.eps_host = inp["eps"] if keep_host_tokens else None
        self.g = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
        del inp
        g = self.g
        self.act = "swiglu" if w.act == W.ACT_SWIGLU else "gelu"
        self.C = api.capacity(w.T, w.k, w.E, w.capacity_factor)
        sw = W.shared_wide(g)
        self.Fsh = 0 if sw["W1s"] is None else sw["W1s"].shape[0]
        self.shape = api.shape_of(w.T, w.d, w.E, w.k, w.F, w.dtype, self.act, d_ff_shared=self.Fsh,
                                  routing=w.routing)
        self.shared_t = None
        self.shared_w = None
        if self.Fsh:
            b2s = None if sw["b2s_rows"] is None else sw["b2s_rows"].sum(dim=0).contiguous()
            self.shared_t = dict(W1s=sw["W1s"], W2s=sw["W2s"], W3s=sw["W3s"], b1s=sw["b1s"], b2s=b2s)
            self.shared_w = api.shared_weights(**self.shared_t)
        self.shared_arg = ctypes.addressof(self.shared_w) if self.shared_w is not None else None
        self.ws = api.new_workspace(self.shape, self.C, dev)
        self.out = torch.empty(w.T, w.d, dtype=w.dtype, device=dev)
        self.counts = torch.empty(w.E, dtype=torch.int32, device=dev)
        self.dropped = torch.empty(1, dtype=torch.int64, device=dev)

    def args(self, stats=None, idx=None, logits=None):
        import ctypes

        import torch

        from sparse_mixture_experts_51_b300 import api
        P, g, w = api._ptr, self.g, self.w
        # the stream current at the call (the capture stream while a graph is recorded)
        sptr = ctypes.c_void_p(torch.cuda.current_stream(self.dev).cuda_stream)
        return [ctypes.byref(self.shape), float(w.capacity_factor), -1, P(g["x"]), P(g["W_g"]), P(g["b_g"]),
                P(g["W_noise"]), P(g["eps"]), P(g["W1"]), P(g["W3"]), P(g["W2"]), P(g["b1"]), P(g["b2"]),
                self.shared_arg, P(self.out), None, P(idx), None, None, P(self.counts), None, P(self.dropped),
                P(stats), P(logits), P(self.ws), self.ws.numel(), sptr]

    def forward(self, **kw):
        from sparse_mixture_experts_51_b300 import _lib
        _lib.check(self.lib.moe_forward(*self.args(**kw)), "moe_forward")

    def forward_timed(self, events):
        import ctypes

        from sparse_mixture_experts_51_b300 import _lib
        arr = (ctypes.c_void_p * 6)(*[None if e is None else ctypes.c_void_p(e.cuda_event) for e in events])
        _lib.check(self.lib.moe_forward_timed(*self.args(), arr), "moe_forward_timed")

    def device_error(self):
        from sparse_mixture_experts_51_b300 import api
        return api.get_device_error(self.ws)


# events of the headline timing: before the router and after the combine
# only.  An event recorded between two kernels cuts their overlap
# (programmatic dependent launch lets a kernel start while its predecessor
# finishes, and the decode-sized layer's expert FFN start while the routing
# runs), so the spans come from a second, shorter run with events around
# expert GEMM 1 (the roofline kernel)
TIMED_SLOTS = (0, 5)
SPAN_SLOTS = (0, 2, 3, 5)
SPANS = {"router_dispatch_gather": (0, 2), "expert_gemm1": (2, 3), "expert_gemm2_combine": (3, 5)}
SPAN_STEPS = 50
# the per-stage split takes every event (which cuts the overlap between stages)
STAGE_SPANS = {"router": (0, 1), "dispatch_gather": (1, 2), "expert_gemm1": (2, 3), "expert_gemm2": (3, 4),
               "combine": (4, 5)}
GRAPH_STEPS = 250


def time_steps(L, steps, flush, eager=False, slots=TIMED_SLOTS, spans=None, sampler=None, barrier=None):
    """Time ``steps`` layer forwards (moe_forward_timed; CUDA graphs of up to
    GRAPH_STEPS steps, the L2 flush before each step outside its events).
    Returns per-step device times (ms) and the per-step span times."""
    import contextlib

    import torch
    G = min(steps, GRAPH_STEPS)
    evs = [[torch.cuda.Event(enable_timing=True) if i in slots else None for i in range(6)] for _ in range(G)]
    stream = torch.cuda.current_stream(L.dev)
    # every event exists on the device before its handle is used
    for row in evs:
        for e in row:
            if e is not None:
                e.record(stream)
    torch.cuda.synchronize()

    graphs = {}
    chunks = [G] * (steps // G) + ([steps % G] if steps % G else [])
    if not eager:
        for n in set(chunks):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr):
                for i in range(n):
                    flush()
                    L.forward_timed(evs[i])
            torch.cuda.synchronize()
            graphs[n] = gr

    spans = spans or {}
    step_ms, span_ms = [], {k: [] for k in spans}
    with (sampler if sampler is not None else contextlib.nullcontext()):
        if sampler is not None:
            sampler.wait_started()
        if barrier is not None:
            barrier()
        torch.cuda.synchronize()
        for n in chunks:
            if eager:
                for i in range(n):
                    flush()
                    L.forward_timed(evs[i])
            else:
                graphs[n].replay()
            torch.cuda.synchronize()
            step_ms += [row[slots[0]].elapsed_time(row[slots[-1]]) for row in evs[:n]]
            for k, (u, v) in spans.items():
                span_ms[k] += [row[u].elapsed_time(row[v]) for row in evs[:n]]
        if barrier is not None:
            barrier()
        torch.cuda.synchronize()
    return step_ms, span_ms


def roofline_of(L, work, gemm1_ms, step_ms_mean, peaks, long_run):
    """Roofline of the layer's dominant work.  Compute-bound shapes: expert
    GEMM 1's TFLOP/s against the measured bf16 peak (the sustained figure when
    the timed run is long enough for the power cap to set the clock, the burst
    figure otherwise; both fractions are given).  Weight-streaming shapes: the
    whole step's algorithmic HBM bytes over the step time against the measured
    copy bandwidth and the nominal ~8 TB/s."""
    w = L.w
    traffic = recorded_traffic(w.name)
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    kernel = "grouped_gemm_kernel (expert GEMM 1, fused activation)"
    if w.dtype_name != "bf16":
        return {"kernel": "whole layer (fp32 CUDA-core path)", "bound": "latency", "achieved": step_ms_mean * 1e3,
                "unit": "us/step", "peak": None, "frac": None,
                "note": "a 64-token fp32 layer: six launches of a few microseconds each, no roofline applies"}
    if work["gemm1_flops"] / work["gemm1_bytes"] >= ridge:
        ach = work["gemm1_flops"] / (gemm1_ms / 1e3) / 1e12
        peak = peaks["bf16_tflops_sustained"] if long_run else peaks["bf16_tflops"]
        return {"kernel": kernel, "bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                "frac": ach / peak, "peak_source": peaks["source"] + (" bf16 sustained" if long_run else " bf16 burst"),
                "frac_of_burst": ach / peaks["bf16_tflops"], "frac_of_sustained": ach / peaks["bf16_tflops_sustained"],
                "algorithmic_flops": work["gemm1_flops"], "ms_per_launch": gemm1_ms, "traffic": traffic,
                "layer_tflops": work["ffn_flops"] / (step_ms_mean / 1e3) / 1e12}
    ach = work["layer_bytes"] / (step_ms_mean / 1e3) / 1e9
    roof = {"kernel": "whole step (expert weight stream: both expert GEMMs)", "bound": "hbm", "achieved": ach,
            "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": ach / peaks["hbm_gbs"],
            "peak_source": peaks["source"] + " copy bandwidth", "frac_of_nominal_8tbs": ach / HBM_NOMINAL_GBS,
            "algorithmic_bytes": work["layer_bytes"], "weight_bytes": work["weight_bytes"], "traffic": traffic}
    if fused_decode_ffn(w):
        # one kernel runs both expert GEMMs (the span between stage events 2 and 3)
        roof.update({"ffn_kernel": "ffn_decode_kernel (both expert GEMMs, fused)", "ffn_ms": gemm1_ms,
                     "ffn_weight_gbs": work["weight_bytes"] / (gemm1_ms / 1e3) / 1e9})
    else:
        roof.update({"gemm1_gbs": work["gemm1_bytes"] / (gemm1_ms / 1e3) / 1e9, "gemm1_ms": gemm1_ms})
    return roof


def fused_decode_ffn(w) -> bool:
    """Whether the library runs this layer's expert FFN as its fused decode
    kernel (bf16, token choice, T <= 128 and T*k >= 4E: the rule in
    ffn_decode.cu)."""
    return w.dtype_name == "bf16" and w.routing == "token" and 1 <= w.T <= 128 and w.T * w.k >= 4 * w.E


def e2e_of(L, n_steps, warmup, world=1):
    """End to end through the public API (MoELayer) with host buffers: every
    step copies its tokens (and noise) from pinned host memory, runs the layer
    and reads the output back to pinned host memory.  Like a serving loop the
    steps are pipelined on three streams with two device buffer sets: the
    input copy of step i+1 and the output copy of step i-1 overlap the layer
    of step i.  The timed region spans the first input copy to the last
    output copy; no L2 flush (every step's inputs arrive from the host, and
    the expert weights are read from HBM each step)."""
    import torch

    from sparse_mixture_experts_51_b300 import api
    w, g, dev = L.w, L.g, L.dev
    stream = torch.cuda.current_stream(dev)
    layer = api.MoELayer(g["W_g"], g["W1"], g["W2"], w.k, L.act, W3=g["W3"], b_g=g["b_g"], W_noise=g["W_noise"],
                         b1=g["b1"], b2=g["b2"], capacity_factor=w.capacity_factor, keep_routing=False,
                         routing=w.routing, **(L.shared_t or {}))
    x_host = L.x_host.pin_memory()
    eps_host = L.eps_host.pin_memory() if L.eps_host is not None else None
    out_host = [torch.empty(w.T, w.d, dtype=w.dtype).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(g["x"]) for _ in range(2)]
    eps_dev = [torch.empty_like(g["eps"]) if g["eps"] is not None else None for _ in range(2)]
    out_dev = [torch.empty_like(L.out) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def run(n):
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

    run(max(2, warmup))
    # at least ~100 ms of steps: each timed run also carries a fixed host-side start-up cost
    n = max(2, n_steps)
    probe_ms = run(4) / 4
    n = int(min(5000, max(n, math.ceil(100.0 / max(probe_ms, 1e-3)))))
    ms = max_over_ranks(run(n), world, dev)
    # the layer run through the public call gives the device-timed output, bit for bit
    if not torch.equal(out_host[(n - 1) % 2], L.out.cpu()):
        raise RuntimeError(f"{w.name}: end-to-end output differs from the timed layer's output")
    h2d = x_host.numel() * x_host.element_size() + (eps_host.numel() * 4 if eps_host is not None else 0)
    d2h = out_host[0].numel() * out_host[0].element_size()
    # the host link alone: the same input copy, back to back, timed on its own
    link = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    with torch.cuda.stream(s_in):
        x_dev[0].copy_(x_host, non_blocking=True)
        link[0].record(s_in)
        for _ in range(5):
            x_dev[0].copy_(x_host, non_blocking=True)
        link[1].record(s_in)
    torch.cuda.synchronize()
    link_gbs = 5 * x_host.numel() * x_host.element_size() / (link[0].elapsed_time(link[1]) / 1e3) / 1e9
    return {"value": job_throughput(w.T, n, world, ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": n, "ms_per_step": ms / n,
            "h2d_gbs_achieved": h2d * n / (ms / 1e3) / 1e9, "h2d_gbs_link": link_gbs,
            "pipelined": "input copy of step i+1 and output copy of step i-1 overlap the layer of step i "
                         "(two buffer sets, three streams)"}


def routing_counts(L):
    """One forward with the routing statistics on: [fp64-re-evaluated tokens,
    near-tie tokens (k-th and (k+1)-th logits within 1e-4)], the kept rows per
    expert and the drop count."""
    import torch
    if L.w.routing != "token":
        L.forward()
        torch.cuda.synchronize()
        return None, L.counts.cpu().tolist(), int(L.dropped.item())
    stats = torch.zeros(2, dtype=torch.int64, device=L.dev)
    L.forward(stats=stats)
    torch.cuda.synchronize()
    st = stats.cpu().tolist()
    return {"fp64_reevaluated_tokens": st[0], "near_tie_tokens": st[1],
            "near_tie_rule": "k-th and (k+1)-th fp32 logits within 1e-4 (routing is exact for them too: "
                             "the router certifies its order and re-evaluates unsettled tokens in fp64)"}, \
        L.counts.cpu().tolist(), int(L.dropped.item())


def routing_stats_of(L, peaks):
    """moe_routing_stats (routing diagnostics + aux loss) over the layer's
    batch, timed as a CUDA graph of back-to-back calls: the call follows the
    layer, whose router has just written the logits, so its inputs are
    L2-resident."""
    import ctypes

    import torch

    from sparse_mixture_experts_51_b300 import _lib, api
    w, dev, lib = L.w, L.dev, L.lib
    if w.routing != "token":
        return None
    P = api._ptr
    logits = torch.empty(w.T, w.E, dtype=torch.float32, device=dev)
    idx_t = torch.empty(w.T, w.k, dtype=torch.int32, device=dev)
    L.forward(idx=idx_t, logits=logits)
    st_out = [torch.empty(n, dtype=torch.float64, device=dev) for n in (w.E, w.E, len(api.STATS_SUMMARY))]

    def call():
        sptr = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
        _lib.check(lib.moe_routing_stats(ctypes.byref(L.shape), P(logits), P(idx_t), P(L.counts), P(L.dropped),
                                         P(st_out[0]), P(st_out[1]), P(st_out[2]), P(L.ws), L.ws.numel(), sptr),
                   "moe_routing_stats")

    n_st = 50
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    gst = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gst):
        for _ in range(n_st):
            call()
    stream = torch.cuda.current_stream(dev)
    gst.replay()
    sev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    sev[0].record(stream)
    gst.replay()
    sev[1].record(stream)
    torch.cuda.synchronize()
    if L.device_error() != 0:
        raise RuntimeError("device-side error in moe_routing_stats")
    st_ms = sev[0].elapsed_time(sev[1]) / n_st
    st_bytes = w.T * w.E * 4 + w.T * w.k * 4  # logits + top-k table, read once
    summ = dict(zip(api.STATS_SUMMARY, st_out[2].tolist()))
    return {"us_per_call": st_ms * 1e3, "timing": f"CUDA graph of {n_st} back-to-back calls, inputs L2-resident",
            "algorithmic_bytes": st_bytes, "achieved_gbs": st_bytes / (st_ms / 1e3) / 1e9,
            "frac_hbm": st_bytes / (st_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
            "aux_loss": summ["aux_loss"], "entropy": summ["entropy"], "load_cv": summ["load_cv"],
            "overflow": summ["overflow"]}


def shared_ffn_of(L, flush, peaks):
    """The shared experts alone (moe_shared_ffn: two dense GEMMs over every
    token), kernel time with L2 flushed before each call."""
    import ctypes

    import torch

    from sparse_mixture_experts_51_b300 import _lib, api
    from sparse_mixture_experts_51_b300 import workloads as W
    if not L.Fsh:
        return None
    w, dev, P = L.w, L.dev, api._ptr
    y_sh = torch.empty(w.T, w.d, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call():
        _lib.check(L.lib.moe_shared_ffn(ctypes.byref(L.shape), P(L.g["x"]), L.shared_arg, P(y_sh), P(L.ws),
                                        L.ws.numel(), ctypes.c_void_p(stream.cuda_stream)), "moe_shared_ffn")

    for _ in range(3):
        call()
    n = 50
    hev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for i in range(n):
        flush()
        hev[i][0].record(stream)
        call()
        hev[i][1].record(stream)
    torch.cuda.synchronize()
    if L.device_error() != 0:
        raise RuntimeError("device-side error in moe_shared_ffn")
    ms = statistics.mean(s_.elapsed_time(e_) for s_, e_ in hev)
    flops = 2.0 * w.T * w.d * L.Fsh * ((2 if w.act == W.ACT_SWIGLU else 1) + 1)
    return {"us_per_call": ms * 1e3, "algorithmic_flops": flops, "achieved_tflops": flops / (ms / 1e3) / 1e12,
            "frac_bf16": flops / (ms / 1e3) / 1e12 / peaks["bf16_tflops"],
            "peak_source": peaks["source"] + " bf16 burst", "launches_per_call": 2}


def cpu_baselines(w, budget_s, single_thread):
    """The oracle on all host threads (and on one thread for small layers)."""
    v, sample, cores, _ = cpu_oracle_run(w, budget_s)
    out = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample, "cpu_model": cpu_model()}
    if single_thread:
        v1, sample1, _, _ = cpu_oracle_run(w, budget_s, threads=1)
        out["single_thread"] = {"value": v1, "unit": UNIT, "cores": 1, "sample": sample1}
    return out


def measure(L, a, flush, peaks, steps, e2e_steps, world=1, sampler_index=0, barrier=None):
    """Everything the JSON line reports about one layer."""
    import torch
    w = L.w
    for _ in range(max(3, a.warmup)):
        L.forward()
        flush()
    torch.cuda.synchronize()
    if L.device_error() != 0:
        raise RuntimeError(f"{w.name}: device-side error in the warm-up")
    # kernels one step enqueues (the library counts its own launches; a graph
    # replays exactly what one captured call enqueued)
    n0 = L.lib.moe_kernel_launches()
    L.forward()
    kernels_per_step = int(L.lib.moe_kernel_launches() - n0)
    torch.cuda.synchronize()

    sampler = ClockSampler(sampler_index)
    step_ms, _ = time_steps(L, steps, flush, eager=a.eager, sampler=sampler, barrier=barrier)
    if L.device_error() != 0:
        raise RuntimeError(f"{w.name}: device-side error during the timed region")
    total_ms = max_over_ranks(sum(step_ms), world, L.dev)
    # outside the timed region: the spans around expert GEMM 1, and the
    # per-stage split with every stage event recorded
    _, span_ms = time_steps(L, min(steps, SPAN_STEPS), flush, eager=a.eager, slots=SPAN_SLOTS, spans=SPANS)
    _, stage = time_steps(L, min(steps, 20), flush, eager=a.eager, slots=tuple(range(6)), spans=STAGE_SPANS)
    routing, counts, dropped = routing_counts(L)
    work = layer_work(w, counts)
    mean_step = total_ms / steps
    gemm1_ms = statistics.mean(span_ms["expert_gemm1"])
    long_run = total_ms >= 1000.0
    res = {
        "value": job_throughput(w.T, steps, world, total_ms), "ms_per_step": mean_step, "steps": steps,
        "step_ms_quantiles": step_quantiles(step_ms),
        "stage_ms": {k: statistics.mean(v) for k, v in span_ms.items()},
        "stage_ms_note": (f"a separate run of {min(steps, SPAN_STEPS)} steps with events before the router, "
                          "around expert GEMM 1 and after the combine (the events cut the overlap at those borders)"
                          + ("; expert_gemm1 is the fused decode FFN (both expert GEMMs)" if fused_decode_ffn(w)
                             else "")),
        "stage_split_ms": {k: statistics.mean(v) for k, v in stage.items()},
        "stage_split_note": "every stage event recorded: no programmatic-launch overlap across the stage borders",
        "roofline": roofline_of(L, work, gemm1_ms, mean_step, peaks, long_run),
        "gpu_launches": kernels_per_step * steps, "kernels_per_step": kernels_per_step,
        "clocks": sampler.summary(),
        "run": {"C": L.C, "kept_rows": work["kept_rows"], "active_experts": work["active_experts"],
                "dropped": dropped, "parallelism": "replicas" if world > 1 else "single_gpu",
                "launch": "eager" if a.eager else f"CUDA graphs of up to {GRAPH_STEPS} timed steps "
                                                  "(moe_forward_timed each)"},
        "routing": routing,
        "e2e": e2e_of(L, e2e_steps, a.warmup, world),
    }
    return res


def run_ours(a):
    import torch
    import torch.distributed as dist

    from sparse_mixture_experts_51_b300 import _lib
    from sparse_mixture_experts_51_b300 import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    lib = _lib.load()
    peaks = load_peaks()
    flush = L2Flush(dev)

    w = replica_workload(W.WORKLOADS[a.workload], rank, world)
    L = DeviceLayer(w, dev, lib)
    m = measure(L, a, flush, peaks, a.steps, max(2, a.steps), world, local,
                barrier=(dist.barrier if world > 1 else None))
    routing_stats = routing_stats_of(L, peaks)
    shared_ffn = shared_ffn_of(L, flush, peaks)
    head_out = L.out  # kept for nothing beyond this point
    del L, head_out
    torch.cuda.empty_cache()

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return 0

    cpu = None
    if not a.no_cpu_baseline and world == 1:
        cpu = cpu_baselines(w, a.cpu_seconds, single_thread=w.name in SINGLE_THREAD_CPU)

    # ---------------- every layer configuration, one at a time (one GPU only)
    per_config = None
    if world == 1 and not a.no_per_config and a.workload in PER_CONFIG:
        per_config = {}
        for name in PER_CONFIG:
            if name == a.workload:
                entry = {k: m[k] for k in ("value", "ms_per_step", "steps", "step_ms_quantiles", "stage_ms",
                                           "stage_split_ms", "roofline", "gpu_launches", "clocks", "run",
                                           "routing", "e2e")}
                entry["cpu_baseline"] = cpu
            else:
                wc = W.WORKLOADS[name]
                Lc = DeviceLayer(wc, dev, lib)
                mc = measure(Lc, a, flush, peaks, min(a.steps, PER_CONFIG_STEPS),
                             min(max(2, a.steps), PER_CONFIG_E2E_STEPS), 1, local)
                del Lc
                torch.cuda.empty_cache()
                entry = {k: mc[k] for k in ("value", "ms_per_step", "steps", "step_ms_quantiles", "stage_ms",
                                            "stage_split_ms", "roofline", "gpu_launches", "clocks", "run",
                                            "routing", "e2e")}
                entry["cpu_baseline"] = (None if a.no_cpu_baseline else
                                         cpu_baselines(wc, 3.0, single_thread=name in SINGLE_THREAD_CPU))
            entry["unit"] = UNIT
            entry["us_per_step"] = entry["ms_per_step"] * 1e3
            entry["config"] = workload_config(W.WORKLOADS[name])
            per_config[name] = entry

    line = {"metric": METRIC, "value": m["value"], "unit": UNIT, "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": m["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "step_ms_quantiles": m["step_ms_quantiles"],
            "dtype": w.dtype_name, "data": "synthetic", "config": workload_config(w), "run": m["run"],
            "stage_ms": m["stage_ms"], "stage_split_ms": m["stage_split_ms"], "roofline": m["roofline"],
            "cpu_baseline": cpu, "e2e": m["e2e"], "gpu_launches": m["gpu_launches"], "clocks": m["clocks"],
            "routing": m["routing"], "routing_stats": routing_stats}
    if shared_ffn is not None:
        line["shared_ffn"] = shared_ffn
    if per_config is not None:
        line["per_config"] = per_config
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
