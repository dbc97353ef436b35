"""Throughput of the attention forward pass on GB300, one JSON line.

A step is one forward pass (one kernel launch) over one batch of seeded
synthetic inputs already resident in HBM.  The default workload is causal GQA
attention, B=2, Hq=32, Hkv=8, Sq=Skv=4096, D=128, bf16 -- the configuration
the headline metric (attention forward TFLOP/s, bf16 causal, S=4096, D=128)
is quoted on.  FLOPs per step = 4*B*Hq*Sq*Skv*D, halved for causal.

  python bench.py [--gpus N --steps K --warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle, same metric

For N > 1 (torchrun, one rank per GPU) every rank runs its own replica of the
workload (weak scaling, no collective on the data path); the timed region is
bracketed by barriers and the slowest rank's time is used.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s (bf16 causal, S=4096, D=128) and % of GB300 tensor peak"
L2_BYTES = 129 * 1024 * 1024

# name -> (B, Hq, Hkv, S, D, causal, dtype)
WORKLOADS = {
    "gqa-causal-4096": (2, 32, 8, 4096, 128, True, "bf16"),
    "tiny-mha": (1, 2, 2, 128, 64, False, "bf16"),
    "mha-causal-1024": (4, 16, 16, 1024, 64, True, "bf16"),
    "fp8-causal-8192": (2, 16, 16, 8192, 128, True, "e4m3"),
}
# the codelab's small timing problem (B=4, T=128, N=8) at D = 32 / 64 / 128 and
# its batch sweep at T=256: launch-latency rows
for _D in (32, 64, 128):
    WORKLOADS[f"latency-b4-t128-d{_D}"] = (4, 8, 8, 128, _D, False, "bf16")
for _B in (1, 2, 4, 8, 16):
    WORKLOADS[f"batch-{_B}-t256"] = (_B, 8, 8, 256, 64, False, "bf16")
for _B, _S in [(64, 512), (32, 1024), (16, 2048), (8, 4096), (4, 8192), (2, 16384)]:
    WORKLOADS[f"mqa-causal-{_S}"] = (_B, 32, 1, _S, 128, True, "bf16")
    WORKLOADS[f"mqa-full-{_S}"] = (_B, 32, 1, _S, 128, False, "bf16")
# decode shapes (few query rows, long K/V; non-causal), run through the
# decode pass with a split workspace: name -> (B, Hq, Hkv, Sq, Skv, D)
DECODE_WORKLOADS = {
    "decode-gqa-b8-32k": (8, 32, 8, 1, 32768, 128),
    "decode-gqa-b32-8k": (32, 32, 8, 4, 8192, 128),
}
# backward pass (gradients of sum(dO * O)): name -> (B, Hq, Hkv, S, D, causal[, dtype]);
# "e4m3": the FP8 pass (E4M3 Q, K, V, E5M2 dO) on the FP8 forward's shape
BWD_WORKLOADS = {
    "bwd-gqa-causal-4096": (2, 32, 8, 4096, 128, True),
    "bwd-mqa-causal-4096": (8, 32, 1, 4096, 128, True),
    "bwd-mqa-full-16384": (2, 32, 1, 16384, 128, False),
    "bwd-mha-causal-1024": (4, 16, 16, 1024, 64, True),
    "bwd-fp8-causal-8192": (2, 16, 16, 8192, 128, True, "e4m3"),
}
DEFAULT_WORKLOAD = "gqa-causal-4096"


class Spec(tuple):
    """(B, Hq, Hkv, Sq, Skv, D, causal, dtype, decode) of a workload."""
    __slots__ = ()
    B = property(lambda t: t[0]); Hq = property(lambda t: t[1]); Hkv = property(lambda t: t[2])
    Sq = property(lambda t: t[3]); Skv = property(lambda t: t[4]); D = property(lambda t: t[5])
    causal = property(lambda t: t[6]); dtype = property(lambda t: t[7]); decode = property(lambda t: t[8])


def spec(name):
    if name in BWD_WORKLOADS:
        B, Hq, Hkv, S, D, causal, *dt = BWD_WORKLOADS[name]
        return Spec((B, Hq, Hkv, S, S, D, causal, dt[0] if dt else "bf16", False))
    if name in DECODE_WORKLOADS:
        B, Hq, Hkv, Sq, Skv, D = DECODE_WORKLOADS[name]
        return Spec((B, Hq, Hkv, Sq, Skv, D, False, "bf16", True))
    B, Hq, Hkv, S, D, causal, dtype = WORKLOADS[name]
    return Spec((B, Hq, Hkv, S, S, D, causal, dtype, False))


ALL_WORKLOADS = sorted(list(WORKLOADS) + list(DECODE_WORKLOADS) + list(BWD_WORKLOADS))


def describe(name):
    w = spec(name)
    seq = f"Sq=Skv={w.Sq}" if w.Sq == w.Skv else f"Sq={w.Sq} Skv={w.Skv}"
    kind = "decode pass, " if w.decode else ""
    return (f"{kind}{'causal' if w.causal else 'non-causal'} B={w.B} Hq={w.Hq} Hkv={w.Hkv} {seq} D={w.D} "
            f"{w.dtype}")


def step_flops(name):
    """4 D FLOPs per visible score (causal: the lower triangle, Sq = Skv);
    the backward pass's five products (S, dP, dV, dK, dQ) are 10 D."""
    w = spec(name)
    f = (10.0 if name in BWD_WORKLOADS else 4.0) * w.B * w.Hq * w.Sq * w.Skv * w.D
    return f / 2 if w.causal else f


def step_bytes(name):
    """Algorithmic bytes: Q, K, V read once and O written once (backward:
    Q, K, V, O, dO and the LSE read, dQ, dK, dV written)."""
    w = spec(name)
    if name in BWD_WORKLOADS:
        e = 1 if w.dtype == "e4m3" else 2        # Q, K, V, dO; O and the gradients are 16-bit
        return w.B * w.D * (w.Sq * w.Hq * (2 * e + 4) + w.Skv * w.Hkv * (2 * e + 4)) + 4 * w.B * w.Hq * w.Sq
    e_in = 1 if w.dtype == "e4m3" else 2
    return w.B * w.D * (w.Sq * w.Hq * e_in + 2 * w.Skv * w.Hkv * e_in + w.Sq * w.Hq * 2)


def n_rotating_sets(name):
    """Input sets to rotate through so that together they hold at least twice
    L2 (two at the least)."""
    return int(min(4096, max(2, -(-2 * L2_BYTES // step_bytes(name)))))


def kernel_source_hash(name=None):
    """Hash of the timed kernel's own sources (device code) for workload
    `name`: a stored DRAM traffic figure is used only while they are
    unchanged.  The backward kernel also includes the forward's header."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "scaled_dot_product_05_gb300", "csrc")
    if name in BWD_WORKLOADS:
        files = (("sdpa_bwd_fp8.cuh",) if spec(name).dtype == "e4m3" else ()) + ("sdpa_bwd.cuh", "sdpa_kernel.cuh",
                                                                                 "ptx.cuh")
    else:
        files = ("sdpa_kernel.cuh", "ptx.cuh")
    for f in files:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


# NVIDIA's nominal dense figures for one GB300 GPU (context beside the measured
# peaks): bf16 2.25 PFLOP/s, FP8 4.5 PFLOP/s, HBM3e ~7.9 TB/s
NOMINAL = {"bf16_tflops": 2250.0, "fp8_tflops": 4500.0, "hbm_gbs": 7900.0}
# the headline's timed region (K steps) is repeated until the repeats add up to
# about this long, so that the clock sampler sees the kernel under load
TIMED_TARGET_MS = 300.0


def cpu_model() -> str:
    """Host CPU model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def workload_config(name, world, **extra):
    """The `config` object of a bench line: the workload by name and sizes
    (identical keys for the GPU arm and the reference arm)."""
    w = spec(name)
    kind = "backward pass, " if name in BWD_WORKLOADS else ""
    cfg = {"workload": kind + describe(name), "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq, "Skv": w.Skv, "D": w.D,
           "causal": w.causal, "flops_per_step": step_flops(name), "parallelism": f"replicas x{world}"}
    cfg.update(extra)
    return cfg


def queue_fill_cycles(steps: int) -> int:
    """GPU clock cycles of sleep that cover the host's submission of `steps`
    bracketed launches (~30 us each at ~2 GHz), at most ~20 ms."""
    return int(min(4e7, 6e4 * steps))


def timed_repeats(region_ms: float) -> int:
    """How many times to repeat a K-step timed region of about region_ms."""
    return int(max(1, min(200, math.ceil(TIMED_TARGET_MS / max(region_ms, 1e-3)))))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def stored_traffic(name):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources and this workload; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f)
    e = t.get(name)
    if not e or e.get("kernel_source_hash") != kernel_source_hash(name):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, timestamped."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    PERIOD_MS = 10

    def __init__(self, index):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.PERIOD_MS)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [p for t, p in self.samples if t0 <= t <= t1]
        note = "samples inside the timed region"
        if not inside:
            # region shorter than the sampling period: nearest samples under load
            near = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
            inside = [p for _, p in near]
            note = f"no sample inside the timed region ({self.PERIOD_MS} ms sampling period); nearest samples"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "nvidia-smi unavailable"}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[0]) for p in inside if num(p[0]) is not None]
        mx = [num(p[1]) for p in inside if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "note": note}


# ------------------------------------------------------------- multi-rank ----

def max_over_ranks(x: float, world: int, device) -> float:
    """Slowest rank's value (all-reduce MAX); `device` is the tensor device the
    process group's backend works on (cuda for NCCL, cpu for gloo)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_step: float, world: int, ms_per_step: float) -> float:
    """Weak scaling: every rank runs its own replica of the workload, so the
    job processes world * flops_per_step per (slowest-rank) step time."""
    return world * flops_per_step / (ms_per_step * 1e-3) / 1e12


# --------------------------------------------------------------- CPU leg ----

def host_threads() -> int:
    """Threads for the CPU oracle: every core this process may run on (the
    launcher's OMP_NUM_THREADS=1 for the GPU ranks does not apply to it)."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def oracle_sample(name, seconds_target=12.0, threads=None):
    """Time the fp64 oracle on a seeded sample of output rows of the workload
    (all host cores unless `threads` is given); returns (TFLOP/s, cores,
    description)."""
    threads = host_threads() if threads is None else threads
    import numpy as np
    import oracle
    from sdpa_inputs import make_qkv

    w = spec(name)
    B, Hq, Hkv, Sq, Skv, D, causal, dtype = w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.causal, w.dtype
    x = make_qkv(1000, B, Hq, Hkv, Sq, Skv, D, dtype)
    rng = np.random.default_rng(1001)
    total_rows = B * Sq * Hq

    def flops_of(rows):
        i = (np.asarray(rows) // Hq) % Sq
        vis = np.minimum(i + 1, Skv) if causal else np.full(len(rows), Skv)
        return 4.0 * D * float(vis.sum())

    def run(rows):
        t0 = time.perf_counter()
        oracle.sdpa_reference(x.q, x.k, x.v, causal=causal, dtype=dtype, descales=x.descales, rows=rows,
                              threads=threads)
        return time.perf_counter() - t0

    n = 256
    rows = np.sort(rng.choice(total_rows, size=min(n, total_rows), replace=False))
    dt = run(rows)
    rate = flops_of(rows) / max(dt, 1e-9)
    # size the timed sample to about `seconds_target` seconds of CPU work
    mean_row = flops_of(rows) / len(rows)
    n = int(min(total_rows, max(64, seconds_target * rate / mean_row)))
    rows = np.sort(rng.choice(total_rows, size=n, replace=False))
    dt = run(rows)
    f = flops_of(rows)
    return f / dt / 1e12, oracle.last_threads(), (
        f"{n} of {total_rows} output rows of the workload, uniformly sampled (seed 1001), "
        f"{f / 1e9:.1f} GFLOP in {dt:.1f} s")


def run_reference(args, rank, world):
    name = args.workload
    if rank != 0:
        return 0
    import numpy as np  # noqa: F401
    per_step_target = min(args.cpu_seconds, max(1.0, min(20.0, 90.0 / max(1, args.steps + args.warmup))))
    values = []
    desc, cores = "", 0
    if name in BWD_WORKLOADS:
        # one bounded sample of the backward oracle (several seconds) stands
        # for every step
        tf, cores, desc = oracle_bwd_sample(name)
        values = [tf]
    else:
        for i in range(args.warmup + args.steps):
            tf, cores, desc = oracle_sample(name, seconds_target=per_step_target)
            if i >= args.warmup:
                values.append(tf)
    value = statistics.median(values)
    ms = step_flops(name) / (value * 1e12) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "ms_per_step_source": "extrapolated: the workload's FLOPs at the rate measured on a bounded row sample "
                              "(the whole workload is not run)",
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1))",
        "config": workload_config(name, world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "cpu_model": cpu_model(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------- GPU leg ----

def run_gpu(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from scaled_dot_product_05_gb300 import (decode_workspace_bytes, sdpa_device_error, sdpa_fwd, sdpa_fwd_decode,
                                             sdpa_fwd_fp8)
    from sdpa_inputs import make_qkv

    name = args.workload
    w = spec(name)
    B, Hq, Hkv, Sq, Skv, D, causal, dtype = w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.causal, w.dtype
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()

    # resident input sets used in rotation, enough that together they hold at
    # least twice L2, so a step never finds its inputs in L2 from an earlier
    # step: two seeded sets, the rest device copies of them
    n_sets = n_rotating_sets(name)
    sets = []
    host = None
    for s in range(2):
        x = make_qkv(100 + 17 * rank + s, B, Hq, Hkv, Sq, Skv, D, dtype)
        q, k, v = (t.to(dev) for t in (x.q, x.k, x.v))
        o = torch.empty((B, Sq, Hq, D), dtype=torch.bfloat16 if dtype == "e4m3" else q.dtype, device=dev)
        sets.append((q, k, v, o, x.descales))
        if s == 0:
            host = x
    for s in range(2, n_sets):
        q, k, v, o, ds = sets[s & 1]
        sets.append((q.clone(), k.clone(), v.clone(), torch.empty_like(o), ds))

    # decode pass: one split workspace, reused by the launches (they run in
    # stream order, never at the same time)
    ws = None
    if w.decode:
        ws = torch.empty(max(16, decode_workspace_bytes(B, Hq, Hkv, Sq, Skv, D)), dtype=torch.uint8, device=dev)

    def launch(i, tensors=None, on=None):
        q, k, v, o, ds = tensors if tensors is not None else sets[i % n_sets]
        st = on if on is not None else stream
        if w.decode:
            sdpa_fwd_decode(q, k, v, o, workspace=ws, stream=st)
        elif dtype == "e4m3":
            sdpa_fwd_fp8(q, k, v, o, descale_q=ds[0], descale_k=ds[1], descale_v=ds[2], causal=causal,
                         stream=st)
        else:
            sdpa_fwd(q, k, v, o, causal=causal, stream=st)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for i in range(args.warmup):
        launch(i)
    barrier()

    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # timed region 1: the K steps back to back, as a caller issues them;
    # repeated (each repeat exactly K steps) until ~TIMED_TARGET_MS have been
    # timed, so the clock samples cover the kernel under load; the value is
    # the median repeat, the slowest rank's
    def region1():
        barrier()
        start.record(stream)
        for i in range(args.steps):
            launch(i)
        end.record(stream)
        barrier()
        return start.elapsed_time(end)

    t_wall0 = time.time()
    region_ms = [region1()]
    n_rep = int(max_over_ranks(timed_repeats(region_ms[0]), world, dev))
    for _ in range(n_rep - 1):
        region_ms.append(region1())
    total_ms = max_over_ranks(statistics.median(region_ms), world, dev)
    ms_per_step = total_ms / args.steps
    # timed region 2: the same K steps, each bracketed by its own events on
    # the launching stream (the kernel's launch duration for the roofline);
    # they queue up behind a short GPU sleep, so that each pair of events
    # brackets its kernel alone, without the host's submission gaps
    torch.cuda._sleep(queue_fill_cycles(args.steps))
    for i in range(args.steps):
        ev[i][0].record(stream)
        launch(i)
        ev[i][1].record(stream)
    barrier()
    t_wall1 = time.time()
    kern_ms = [a.elapsed_time(b) for a, b in ev]
    # the same launches captured in one CUDA graph and replayed: launch
    # latency without the Python call (what a graph-capturing caller sees)
    g_launches = min(args.steps, 32)
    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        for i in range(g_launches):
            launch(i, on=cap)
    graph.replay()
    barrier()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(3):
        graph.replay()
    g1.record(stream)
    barrier()
    graph_ms = g0.elapsed_time(g1) / (3 * g_launches)
    del graph
    err = sdpa_device_error()
    if err:
        raise RuntimeError(f"device error word 0x{err:x}")

    # ---- end to end: pinned host inputs -> device -> kernel -> host output --
    # Every step copies its inputs in from pinned host memory and its output
    # back out.  Serial: copy in, kernel, copy out on one stream.  Pipelined:
    # H2D, compute and D2H on three streams over the two device buffer sets,
    # so step i+1's copy in and step i-1's copy out overlap step i's kernel
    # (events keep each buffer set's reuse in order).
    e2e_steps = max(3, min(args.steps, 20))
    hq_, hk_, hv_ = (t.pin_memory() for t in (host.q, host.k, host.v))
    hos = [torch.empty(sets[i][3].shape, dtype=sets[i][3].dtype).pin_memory() for i in range(2)]
    bi = sum(t.numel() * t.element_size() for t in (hq_, hk_, hv_))
    bo = hos[0].numel() * hos[0].element_size()

    def serial_step():
        q, k, v, o, ds = sets[0]
        q.copy_(hq_, non_blocking=True)
        k.copy_(hk_, non_blocking=True)
        v.copy_(hv_, non_blocking=True)
        launch(0, (q, k, v, o, host.descales))
        hos[0].copy_(o, non_blocking=True)

    for _ in range(2):
        serial_step()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        serial_step()
    e1.record(stream)
    barrier()
    e2e_serial_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)

    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    done_k = [torch.cuda.Event() for _ in range(2)]      # kernel on set i finished (inputs free)
    done_o = [torch.cuda.Event() for _ in range(2)]      # copy-out of set i finished (output free)

    def pipelined(nsteps, first, last):
        for i in range(nsteps):
            sidx = i & 1
            q, k, v, o, ds = sets[sidx]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(done_k[sidx])
                elif first is not None and i == 0:
                    first.record(s_in)
                q.copy_(hq_, non_blocking=True)
                k.copy_(hk_, non_blocking=True)
                v.copy_(hv_, non_blocking=True)
                arrived = torch.cuda.Event()
                arrived.record(s_in)
            stream.wait_event(arrived)
            if i >= 2:
                stream.wait_event(done_o[sidx])
            launch(sidx, (q, k, v, o, host.descales))              # descales of the copied data
            done_k[sidx].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done_k[sidx])
                hos[sidx].copy_(o, non_blocking=True)
                done_o[sidx].record(s_out)
        if last is not None:
            last.record(s_out)

    pipelined(4, None, None)
    barrier()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pipelined(e2e_steps, p0, p1)
    barrier()
    e2e_ms = p0.elapsed_time(p1) / e2e_steps
    # both buffer sets now hold results of the same host inputs
    if not torch.equal(hos[0], hos[1]) or not torch.equal(hos[0], sets[0][3].cpu()):
        raise RuntimeError("pipelined end-to-end outputs disagree")
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    if sampler:
        sampler.stop()

    if rank != 0:
        return 0

    flops = step_flops(name)
    value = whole_job_tflops(flops, world, ms_per_step)
    peaks, peak_src = load_peaks()
    avg_kernel_ms = statistics.mean(kern_ms)
    achieved = flops / (avg_kernel_ms * 1e-3) / 1e12
    if dtype == "e4m3":
        peak = peaks["bf16_tflops"] * 2.0       # FP8 dense rate is twice bf16's (4.5 vs 2.25 PF nominal)
        peak_note = f"bf16 burst ({peak_src}) x 2 nominal FP8/bf16 ratio"
        nominal_tensor = NOMINAL["fp8_tflops"]
        sustained = peaks["bf16_tflops_sustained"] * 2.0
    else:
        peak = peaks["bf16_tflops"]
        peak_note = f"bf16 burst ({peak_src})"
        nominal_tensor = NOMINAL["bf16_tflops"]
        sustained = peaks["bf16_tflops_sustained"]
    achieved_gbs = step_bytes(name) / (avg_kernel_ms * 1e-3) / 1e9
    # the bound is whichever roofline time is longer: FLOPs at the tensor peak
    # or algorithmic bytes at the HBM peak
    t_tensor = flops / (peak * 1e12)
    t_hbm = step_bytes(name) / (peaks["hbm_gbs"] * 1e9)
    if t_hbm > t_tensor:
        roofline = {"bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": achieved_gbs / peaks["hbm_gbs"], "traffic": stored_traffic(name),
                    "peak_source": f"HBM copy ({peak_src})", "nominal_peak": NOMINAL["hbm_gbs"],
                    "frac_of_nominal": achieved_gbs / NOMINAL["hbm_gbs"], "achieved_tflops": achieved,
                    "tensor_peak_tflops": peak}
    else:
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": stored_traffic(name), "peak_source": peak_note,
                    "sustained_peak": sustained, "frac_of_sustained": achieved / sustained,
                    "nominal_peak": nominal_tensor, "frac_of_nominal": achieved / nominal_tensor,
                    "achieved_hbm_gbs": achieved_gbs, "hbm_peak_gbs": peaks["hbm_gbs"]}
    roofline.update({"kernel": "sdpa_fwd_kernel", "algorithmic_bytes_per_launch": step_bytes(name),
                     "roofline_time_ms": max(t_tensor, t_hbm) * 1e3,
                     "frac_of_roofline_time": max(t_tensor, t_hbm) * 1e3 / avg_kernel_ms})
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": dtype, "data": "synthetic (seeded N(0,1), inputs resident in HBM)",
        "config": workload_config(name, world,
                                  l2=f"inputs larger than L2 ({n_sets} rotating input sets of "
                                     f"{step_bytes(name) / 1e6:.1f} MB, {n_sets * step_bytes(name) / 1e6:.0f} MB in all)",
                                  timed_region=f"{len(region_ms)} repeats of the {args.steps} steps (median repeat; "
                                               f"{sum(region_ms):.0f} ms timed in all)"),
        "roofline": roofline,
        "e2e": {"value": whole_job_tflops(flops, world, e2e_ms), "unit": "TFLOP/s", "h2d_bytes_per_step": bi,
                "d2h_bytes_per_step": bo, "ms_per_step": e2e_ms,
                "pipelined": "H2D / kernel / D2H on three streams over two device buffer sets",
                "serial_ms_per_step": e2e_serial_ms,
                "serial_value": whole_job_tflops(flops, world, e2e_serial_ms)},
        "gpu_launches": (len(region_ms) + 1) * args.steps,
        "graph": {"ms_per_launch": graph_ms, "launches": 3 * g_launches,
                  "note": "the same launches captured in one CUDA graph and replayed (no Python call per launch); "
                          "timed regions 1 (back to back, gives value) and 2 (per-launch events, gives the "
                          "roofline's launch duration) hold K launches each"},
        "clocks": sampler.summary(t_wall0, t_wall1) if sampler else None,
    }
    if line["clocks"] and line["clocks"].get("sm_mhz"):
        # time x clock: the work in SM cycles per step, comparable across runs at different clocks
        line["clocks"]["ms_x_mhz_per_step"] = ms_per_step * line["clocks"]["sm_mhz"]
    if not args.no_cpu_baseline:
        tf, cores, desc = oracle_sample(name, seconds_target=args.cpu_seconds)
        tf1, _, desc1 = oracle_sample("tiny-mha", seconds_target=2.0, threads=1)
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": cores, "cpu_model": cpu_model(),
                                "kind": "oracle", "sample": desc,
                                "single_thread": {"workload": describe("tiny-mha"), "value": tf1, "unit": "TFLOP/s",
                                                  "cores": 1, "sample": desc1}}
    print(json.dumps(line), flush=True)
    return 0


def oracle_bwd_sample(name, threads=None):
    """Time the fp64 backward oracle on a bounded sample of the workload:
    batch 0, every KV head (the oracle runs one thread per KV head), the
    first S positions, S a multiple of 256 chosen for about 7.5e9 FLOP per
    thread it gets (10 to 20 s); returns (TFLOP/s, threads, description)."""
    import oracle
    from sdpa_inputs import make_qkv

    threads = host_threads() if threads is None else threads
    w = spec(name)
    per_s2 = 10.0 * w.Hq * w.D * (0.5 if w.causal else 1.0)
    target = 7.5e9 * min(w.Hkv, os.cpu_count() or 1)
    S = max(256, min(w.Sq, int((target / per_s2) ** 0.5) // 256 * 256))
    x = make_qkv(1000, 1, w.Hq, w.Hkv, S, S, w.D, "bf16")
    do = make_qkv(1001, 1, w.Hq, w.Hkv, S, S, w.D, "bf16").q
    t0 = time.perf_counter()
    oracle.sdpa_backward_reference(x.q, x.k, x.v, do, causal=w.causal, dtype="bf16", threads=threads)
    dt = time.perf_counter() - t0
    f = 10.0 * w.Hq * S * S * w.D * (0.5 if w.causal else 1.0)
    return f / dt / 1e12, oracle.last_threads(), (
        f"batch 0, all {w.Hkv} KV heads, positions 0..{S - 1} of the workload: {f / 1e9:.1f} GFLOP in {dt:.1f} s")


def run_gpu_bwd(args, rank, world, local_rank):
    """The backward pass: one step is sdpa_bwd on resident Q, K, V, O, dO and
    the forward's LSE (rotating input sets, as for the forward)."""
    import torch
    import torch.distributed as dist

    from scaled_dot_product_05_gb300 import (bwd_fp8_workspace_bytes, bwd_workspace_bytes, sdpa_bwd, sdpa_bwd_fp8,
                                              sdpa_device_error, sdpa_fwd_ex, sdpa_fwd_fp8_ex)
    from sdpa_inputs import E5M2_MAX, make_grad, make_qkv

    name = args.workload
    w = spec(name)
    B, Hq, Hkv, S, D, causal = w.B, w.Hq, w.Hkv, w.Sq, w.D, w.causal
    fp8 = w.dtype == "e4m3"
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    n_sets = n_rotating_sets(name)
    sets = []
    host = None
    descales = []                    # FP8: (dq, dk, dv, ddo, scale_ds) per set
    for i in range(n_sets):
        if fp8:
            x = make_qkv(100 + 17 * rank + i, B, Hq, Hkv, S, S, D, "e4m3")
            do, ddo = make_grad(200 + 17 * rank + i, (B, S, Hq, D), "e5m2")
        else:
            x = make_qkv(100 + 17 * rank + i, B, Hq, Hkv, S, S, D, "bf16")
            do = make_grad(200 + 17 * rank + i, (B, S, Hq, D), "bf16")
        q, k, v, g = (t.to(dev) for t in (x.q, x.k, x.v, do))
        o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=dev)
        if fp8:
            sdpa_fwd_fp8_ex(q, k, v, o, lse, descale_q=x.descales[0], descale_k=x.descales[1],
                            descale_v=x.descales[2], causal=causal)
            grads = tuple(torch.empty(t.shape, dtype=torch.bfloat16, device=dev) for t in (q, k, v))
        else:
            sdpa_fwd_ex(q, k, v, o, lse, causal=causal)
            grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
        sets.append((q, k, v, o, g, lse, grads))
        if fp8:
            # the recipe's delayed scale of dS: amax of a first call
            amax = torch.zeros(1, dtype=torch.float32, device=dev)
            sdpa_bwd_fp8(q, k, v, o, g, lse, *grads, descale_q=x.descales[0], descale_k=x.descales[1],
                         descale_v=x.descales[2], descale_do=ddo, scale_ds=1.0, amax_ds=amax, causal=causal)
            descales.append((*x.descales, ddo, E5M2_MAX / float(amax.item())))
        if i == 0:
            host = tuple(t.cpu().pin_memory() for t in (q, k, v, o, g, lse))
    ws_bytes = bwd_fp8_workspace_bytes(B, Hq, S, D) if fp8 else bwd_workspace_bytes(B, Hq, S, D)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)

    def launch(i, st=None):
        q, k, v, o, g, lse, (dq, dk, dv) = sets[i % n_sets]
        if fp8:
            a, b_, c, d, sds = descales[i % n_sets]
            sdpa_bwd_fp8(q, k, v, o, g, lse, dq, dk, dv, descale_q=a, descale_k=b_, descale_v=c, descale_do=d,
                         scale_ds=sds, causal=causal, workspace=ws, stream=st or stream)
        else:
            sdpa_bwd(q, k, v, o, g, lse, dq, dk, dv, causal=causal, workspace=ws, stream=st or stream)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for i in range(args.warmup):
        launch(i)
    barrier()
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        time.sleep(0.3)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def region1():
        barrier()
        start.record(stream)
        for i in range(args.steps):
            launch(i)
        end.record(stream)
        barrier()
        return start.elapsed_time(end)

    t_wall0 = time.time()
    region_ms = [region1()]
    n_rep = int(max_over_ranks(timed_repeats(region_ms[0]), world, dev))
    for _ in range(n_rep - 1):
        region_ms.append(region1())
    ms_per_step = max_over_ranks(statistics.median(region_ms), world, dev) / args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda._sleep(queue_fill_cycles(args.steps))     # the launches queue up behind it
    for i in range(args.steps):
        ev[i][0].record(stream)
        launch(i)
        ev[i][1].record(stream)
    barrier()
    t_wall1 = time.time()
    kern_ms = [a.elapsed_time(b) for a, b in ev]
    err = sdpa_device_error()
    if err:
        raise RuntimeError(f"device error word 0x{err:x}")
    # end to end: inputs copied in from pinned host memory, gradients copied
    # out, every step (serial on the launching stream)
    hq_, hk_, hv_, ho_, hg_, hl_ = host
    out_host = tuple(torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in sets[0][6])
    bi = sum(t.numel() * t.element_size() for t in host)
    bo = sum(t.numel() * t.element_size() for t in out_host)
    q, k, v, o, g, lse, grads = sets[0]
    e2e_steps = max(3, min(args.steps, 10))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    for _ in range(e2e_steps):
        for dst, src in zip((q, k, v, o, g, lse), host):
            dst.copy_(src, non_blocking=True)
        launch(0)
        for dst, src in zip(out_host, grads):
            dst.copy_(src, non_blocking=True)
    e1.record(stream)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)
    if sampler:
        sampler.stop()
    if rank != 0:
        return 0

    flops = step_flops(name)
    peaks, peak_src = load_peaks()
    avg_kernel_ms = statistics.mean(kern_ms)
    achieved = flops / (avg_kernel_ms * 1e-3) / 1e12
    # FP8: twice the measured bf16 peak (the nominal dense FP8 / bf16 ratio)
    peak = peaks["bf16_tflops"] * (2 if fp8 else 1)
    peak_note = f"2 x bf16 burst ({peak_src}), the nominal FP8 / bf16 ratio" if fp8 else f"bf16 burst ({peak_src})"
    nominal_tensor = NOMINAL["fp8_tflops" if fp8 else "bf16_tflops"]
    sustained = peaks["bf16_tflops_sustained"] * (2 if fp8 else 1)
    line = {
        "metric": METRIC, "value": whole_job_tflops(flops, world, ms_per_step), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 x e5m2 (fp32 accumulate)" if fp8 else "bf16",
        "data": "synthetic (seeded N(0,1), inputs resident in HBM)",
        "config": workload_config(name, world,
                                  l2=f"inputs larger than L2 ({n_sets} rotating input sets of "
                                     f"{step_bytes(name) / 1e6:.1f} MB)",
                                  timed_region=f"{len(region_ms)} repeats of the {args.steps} steps (median repeat; "
                                               f"{sum(region_ms):.0f} ms timed in all)"),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                     "traffic": stored_traffic(name), "peak_source": peak_note, "sustained_peak": sustained,
                     "frac_of_sustained": achieved / sustained, "nominal_peak": nominal_tensor,
                     "frac_of_nominal": achieved / nominal_tensor,
                     "kernel": ("sdpa_bwd_fp8_kernel" if fp8 else "sdpa_bwd_kernel") + " (+ Delta, "
                     "dQ conversion; launch duration of the whole call)",
                     "algorithmic_bytes_per_launch": step_bytes(name)},
        "e2e": {"value": whole_job_tflops(flops, world, e2e_ms), "unit": "TFLOP/s", "h2d_bytes_per_step": bi,
                "d2h_bytes_per_step": bo, "ms_per_step": e2e_ms, "pipelined": "no (serial copy in, pass, copy out)"},
        "gpu_launches": (len(region_ms) + 1) * args.steps * 3,
        "clocks": sampler.summary(t_wall0, t_wall1) if sampler else None,
    }
    if line["clocks"] and line["clocks"].get("sm_mhz"):
        line["clocks"]["ms_x_mhz_per_step"] = ms_per_step * line["clocks"]["sm_mhz"]
    if not args.no_cpu_baseline and world == 1:
        tf, cores, desc = oracle_bwd_sample(name)
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": cores, "cpu_model": cpu_model(),
                                "kind": "oracle", "sample": desc}
    print(json.dumps(line), flush=True)
    return 0


def launch_command(n_gpus, argv):
    """The torchrun command line that runs this script with `argv` as one
    rank per GPU on this node (rendezvous on 127.0.0.1, a free port)."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n_gpus}",
            "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *argv]


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=ALL_WORKLOADS, default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        # one process per GPU: start this same command under torchrun
        os.execv(sys.executable, launch_command(args.gpus, sys.argv[1:]))
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}", file=sys.stderr)
        return 2
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        if args.workload in BWD_WORKLOADS:
            return run_gpu_bwd(args, rank, world, local_rank)
        return run_gpu(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
