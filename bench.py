#!/usr/bin/env python3
"""Benchmark: attention forward + backward TFLOP/s on GB300.

One step = one forward (attn_fwd) and one backward (attn_bwd: preprocess,
main, dQ conversion) over one batch of the workload, inputs resident in HBM.
Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload long]
  python bench.py --impl reference ...   # the fp64 CPU oracle, bounded sample

FLOP convention: forward 4*B*H*N^2*d (halved when causal), backward 2.5x
forward.  Multi-GPU (torchrun): every rank runs the same workload on its own
GPU (independent replicas: attention over (b, h) needs no exchange), value =
all ranks' FLOPs / max-over-ranks time ("weak" scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import re
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("attn fwd+bwd TFLOP/s (bf16, causal, N=2k–32k) and % of GB300 dense "
          "BF16 peak")
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


BWD_MAIN_SOURCES = ("attn_bwd.cu", "sm103_ptx.cuh", "kernels.h", "dropout.cuh")


def kernel_source_hash(files=BWD_MAIN_SOURCES):
    """sha256 over the sources compiled into the backward main kernel."""
    h = hashlib.sha256()
    for fn in files:
        with open(os.path.join(ROOT, "exact_tiled_attention_22_gb300", "csrc", fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def bwd_main_traffic(workload):
    """DRAM bytes (read + write) per launch of the backward main kernel, from
    the ncu summary under profiles/ -- only if that capture was taken on this
    workload with the sources as they are now, else None."""
    path = os.path.join(ROOT, "profiles", f"attn_bwd_main_{workload}_dram.md")
    try:
        with open(path) as f:
            text = f.read()
    except OSError:
        return None
    fields = dict(re.findall(r"^- ([a-z0-9 ]+): `([^`]+)`", text, flags=re.M))
    if fields.get("source sha256") != kernel_source_hash():
        return None
    try:
        return int(fields["dram bytes per launch"])
    except (KeyError, ValueError):
        return None


def kept_pairs(mask, N, causal):
    """Number of (query, key) scores a [H, nb, nb] block mask keeps, summed
    over heads, with the causal rule key <= query when `causal`."""
    import numpy as np
    m = mask.numpy().astype(bool)
    nb = m.shape[1]
    size = np.minimum(128, N - 128 * np.arange(nb)).astype(np.int64)  # rows per block
    full = np.outer(size, size)
    if causal:
        lower = np.tril(np.ones((nb, nb), dtype=bool), -1)
        tri = size * (size + 1) // 2
        per = np.where(lower, full, 0) + np.diag(tri)
    else:
        per = full
    return int((m * per[None]).sum())


def peak_label(src: str, dtype: str) -> str:
    """The dense tensor peak used for a contraction of `dtype`: the measured
    bf16 burst rate; fp16 takes it too (the nominal fp16 : bf16 dense ratio
    of the tensor cores is 1)."""
    if dtype == "fp16":
        return f"{src} bf16_tflops (burst) x 1 (nominal fp16 : bf16 dense ratio)"
    return f"{src} bf16_tflops (burst)"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------- clocks
class NvmlClocks:
    """SM clock and clock-event reasons read through NVML (ctypes, read-only
    queries) every ~2 ms from a thread, so that a timed region of a few tens
    of milliseconds still gets many samples.  None of the calls changes a
    setting of the GPU."""
    # clock-event reason bits of the NVML API
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap"}

    def __init__(self, uuid: str):
        import ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        self.c = ctypes
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.dev = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.dev)) != 0:
            raise OSError("no NVML device for " + uuid)
        self.fn_reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        self.max_mhz = (float(mx.value) if self.lib.nvmlDeviceGetMaxClockInfo(self.dev, 1, ctypes.byref(mx)) == 0
                        else None)
        self.samples = []  # (monotonic time, SM MHz, reason bits)
        self.stop_flag = False
        self.thread = threading.Thread(target=self._run, daemon=True)

    def _run(self):
        c = self.c
        mhz, rs = c.c_uint(), c.c_ulonglong()
        while not self.stop_flag:
            if (self.lib.nvmlDeviceGetClockInfo(self.dev, 1, c.byref(mhz)) == 0 and
                    self.fn_reasons(self.dev, c.byref(rs)) == 0):
                self.samples.append((time.monotonic(), float(mhz.value), int(rs.value)))
            time.sleep(0.002)

    def start(self):
        self.thread.start()

    def stop(self, t0, t1):
        self.stop_flag = True
        self.thread.join(timeout=2)
        self.lib.nvmlShutdown()
        inside = [x for x in self.samples if t0 <= x[0] <= t1]
        if not inside:
            return None
        reasons = sorted({n for _, _, r in inside for bit, n in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(x[1] for x in inside),
                "sm_max_mhz": self.max_mhz if self.max_mhz else max(x[1] for x in inside),
                "reasons": reasons, "samples": len(inside), "source": "nvml, every ~2 ms"}


class ClockSampler:
    """Clocks and throttle reasons during the timed region: NVML samples
    taken between begin() and end() when NVML can be loaded, else nvidia-smi
    every 100 ms around the region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str, uuid: str = None):
        self.gpu = gpu_id
        self.proc = None
        self.lines = []
        self.thread = None
        self.nvml = None
        self.t0 = self.t1 = None
        if uuid:
            try:
                self.nvml = NvmlClocks(uuid)
            except (OSError, AttributeError):
                self.nvml = None

    def start(self):
        if self.nvml:
            self.nvml.start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def begin(self):
        self.t0 = time.monotonic()

    def end(self):
        self.t1 = time.monotonic()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.nvml:
            t1 = self.t1 if self.t1 is not None else time.monotonic()
            return self.nvml.stop(self.t0 if self.t0 is not None else 0.0, t1)
        if not self.proc:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm),
                "source": "nvidia-smi every 100 ms, from 0.3 s before to 0.15 s after the region"}


def gpu_local_cpus(uuid: str):
    """The CPUs of this process's allowed set that NVML reports as closest to
    the GPU (a read-only query), or None when NVML or the query is not
    available or the sets do not intersect."""
    import ctypes
    try:
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            return None
        try:
            dev = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(dev)) != 0:
                return None
            n = 16  # 16 x 64 CPUs
            mask = (ctypes.c_ulong * n)()
            if lib.nvmlDeviceGetCpuAffinity(dev, n, mask) != 0:
                return None
        finally:
            lib.nvmlShutdown()
    except (OSError, AttributeError):
        return None
    near = {64 * i + b for i in range(n) for b in range(64) if (mask[i] >> b) & 1}
    allowed = os.sched_getaffinity(0)
    both = near & allowed
    return both or None


class on_cpus:
    """Runs the block on the given CPUs (None: unchanged) and restores the
    process's CPU set afterwards.  Pinned host buffers allocated inside are
    first touched there, which puts their pages on the memory next to those
    CPUs: the GPU's, when the CPUs are gpu_local_cpus()."""

    def __init__(self, cpus):
        self.cpus = cpus
        self.prev = None

    def __enter__(self):
        if self.cpus:
            self.prev = os.sched_getaffinity(0)
            os.sched_setaffinity(0, self.cpus)
        return self

    def __exit__(self, *exc):
        if self.prev is not None:
            os.sched_setaffinity(0, self.prev)
        return False


def gpu_uuid(dev) -> str:
    """NVML UUID string ("GPU-...") of a torch CUDA device, or None."""
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
    except (AttributeError, RuntimeError):
        return None
    return u if u.startswith("GPU-") else "GPU-" + u


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time: every rank's step time is all-reduced with MAX
    (NCCL on GPUs, gloo in the CPU tests)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(flops_per_rank: float, world: int, step_ms: float) -> float:
    """Whole-job throughput: every rank's FLOPs over the slowest rank's time."""
    return world * flops_per_rank / (step_ms * 1e-3) / 1e12


def smi_id(local: int) -> str:
    """nvidia-smi --id for this process's GPU (index or UUID)."""
    cvd = os.environ.get("CUDA_VISIBLE_DEVICES", "").strip()
    if cvd:
        ids = [s.strip() for s in cvd.split(",") if s.strip()]
        if local < len(ids):
            return ids[local]
    return str(local)


# ----------------------------------------------------------------- oracle leg
_SAMPLE_INPUTS = {}


def oracle_sample(w, target_s: float):
    """Times the fp64 CPU oracle (as it stands) on heads of the workload's own
    inputs: a causal prefix of head (0, 0), sized for ~target_s of CPU work
    (for a causal workload the first n query rows attend only to the first n
    keys, so the prefix is an exact sub-problem); when a whole head takes
    less than that, further whole heads until about target_s.
    Returns (TFLOP/s, seconds, n, threads, heads)."""
    import oracle
    from exact_tiled_attention_22_gb300.inputs import workload_inputs
    orc = oracle.get()
    threads = orc.threads()
    if w.name not in _SAMPLE_INPUTS:  # drawn once per workload, outside the timing
        _SAMPLE_INPUTS[w.name] = workload_inputs(w)
    x = _SAMPLE_INPUTS[w.name]
    order = [(b, h) for b in range(w.B) for h in range(w.H)]

    def run(n, b, h):
        q, k, v, do = (x[s][b, :n, h, :].double().numpy() for s in ("q", "k", "v", "do"))
        t0 = time.perf_counter()
        orc.fwd_head(q, k, v, w.scale, w.causal, nthreads=threads)
        orc.bwd_head(q, k, v, do, w.scale, w.causal, nthreads=threads)
        dt = time.perf_counter() - t0
        f = 4.0 * n * n * w.d * (0.5 if w.causal else 1.0) * 3.5
        return f, dt

    n = min(w.N, 1024)
    f, dt = run(n, 0, 0)
    if dt < target_s and n < w.N:
        n = min(w.N, int(n * math.sqrt(target_s / max(dt, 1e-3))) // 64 * 64 or 64)
        f, dt = run(n, 0, 0)
    heads = 1
    while n == w.N and dt < 0.8 * target_s and heads < len(order):
        f1, dt1 = run(n, *order[heads])
        f, dt, heads = f + f1, dt + dt1, heads + 1
    return f / dt / 1e12, dt, n, threads, heads


def sample_text(w, n, heads, dt=None):
    took = "" if dt is None else f", {dt:.1f} s"
    if n < w.N:
        return (f"causal prefix of head (0, 0): first {n} query rows/keys, d={w.d}, "
                f"fwd+bwd fp64{took}")
    return f"{heads} whole head(s) (N={n}, d={w.d}) of the workload's inputs, fwd+bwd fp64{took}"


def reference_arm(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    per_step = max(0.5, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    vals = []
    n_used, threads = None, None
    for i in range(args.warmup + args.steps):
        v, dt, n, threads, heads = oracle_sample(w, per_step)
        n_used = (n, heads)
        if i >= args.warmup:
            vals.append((v, dt))
    value = statistics.median(v for v, _ in vals)
    ms = statistics.median(dt for _, dt in vals) * 1e3
    sample = sample_text(w, *n_used)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(w, args),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_dict(w, args=None, kept_fraction=None):
    """The workload's config, the same keys in both arms: the variant keys
    (alibi, block_mask, dropout) are None when the variant is off."""
    alibi = bool(args and args.alibi)
    block_mask = args.block_mask if args else None
    dropout = (args.dropout or None) if args else None
    return {"workload": f"{w.name}: B={w.B} H={w.H} N={w.N} d={w.d} {w.dtype} "
                        f"{'causal' if w.causal else 'non-causal'}",
            "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal, "scale": w.scale,
            "input_dtype": w.dtype,
            "l2": "inputs larger than L2: Q,K,V,O,dO,dQ,dK,dV plus the fp32 dQ accumulator "
                  "exceed 129 MB per step; no flush",
            "alibi": "slopes 2^(-8(h+1)/H)" if alibi else None,
            "block_mask": (None if not block_mask else
                           {"pattern": block_mask, "kept_fraction_of_dense": kept_fraction}),
            "dropout": dropout}


# ----------------------------------------------------------------- our arm
def decode_main(args, w):
    """Decoding against a KV cache (attn_decode): HBM-bound, measured in GB/s
    of K and V streamed from HBM per step.  One step = one attn_decode call;
    the 4.3 GB cache of the default shapes is far larger than L2."""
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps({"impl": "reference", "unavailable":
                              "the decode workloads have no reference arm; the oracle is timed "
                              "in cpu_baseline"}))
        return 0

    from exact_tiled_attention_22_gb300 import build
    build.build()
    from exact_tiled_attention_22_gb300 import attn
    from exact_tiled_attention_22_gb300.inputs import make_decode_inputs

    B, H, Nq, Nk, d = w.B, w.H, w.Nq, w.Nk, w.d
    x = make_decode_inputs(w)
    q_host = x["q"].pin_memory()
    q = q_host.to(dev)
    k, v = x["k"].to(dev), x["v"].to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
    ws = torch.empty(attn.attn_decode_workspace_size(B, H, Nq, Nk, d), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        attn.check(attn.attn_decode(q, k, v, o, lse, B, H, Nq, Nk, d, w.scale, w.causal, w.dtype,
                                    ws, ws.numel(), stream))

    for _ in range(args.warmup):
        step()
    attn.check(attn.attn_status(stream))
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(smi_id(local), gpu_uuid(dev)) if rank == 0 else None
    if sampler:
        sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.begin()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.end()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    attn.check(attn.attn_status(stream))
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / args.steps
    # per-kernel durations: the same steps again with the library's events
    # (not in the timed region: they end the launches' programmatic overlap)
    attn.check(attn.attn_profile_begin())
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize(dev)
    prof = attn.attn_profile_end()
    attn.check(attn.attn_status(stream))
    gpu_launches = sum(n for n, _ in prof.values())

    # end to end: the new query rows in from pinned host memory, O and LSE out
    o_host = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    lse_host = torch.empty(lse.shape, dtype=torch.float32).pin_memory()

    def e2e_step():
        q.copy_(q_host, non_blocking=True)
        step()
        o_host.copy_(o, non_blocking=True)
        lse_host.copy_(lse, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(dev)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    f1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(f0.elapsed_time(f1), world, dev) / args.e2e_steps

    peaks, peak_src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    gbs = w.kv_bytes() * world / (ms * 1e-3) / 1e9
    split_ms = prof["attn_decode_split"][1] / max(1, prof["attn_decode_split"][0])
    split_gbs = w.kv_bytes() / (split_ms * 1e-3) / 1e9

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        import oracle
        orc = oracle.get()
        qs = x["q"][0, :, 0, :].double().numpy()
        ks, vs = (x[n][0, :, 0, :].double().numpy() for n in ("k", "v"))
        t0 = time.perf_counter()
        heads = 0
        while time.perf_counter() - t0 < 5.0 or heads == 0:
            orc.decode_head(qs, ks, vs, w.scale, w.causal, nthreads=orc.threads())
            heads += 1
        dt = time.perf_counter() - t0
        per_head = 2 * w.Nk * w.d * 2
        cpu = {"value": per_head * heads / dt / 1e9, "unit": "GB/s", "cores": orc.threads(),
               "kind": "oracle", "sample": f"head (0, 0), Nq={w.Nq}, Nk={w.Nk}, fp64, "
                                           f"{heads} repetitions in {dt:.1f} s"}

    if rank == 0:
        line = {
            "metric": "attn decode: K/V cache streamed from HBM, GB/s", "value": gbs,
            "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic",
            "config": dict(w.as_dict(), l2="K/V cache (4.3 GB) far larger than L2; no flush"),
            "kernel_ms": {nm: (t / n if n else None) for nm, (n, t) in prof.items() if n},
            "roofline": {"kernel": "attn_decode_split", "bound": "hbm", "achieved": split_gbs,
                         "peak": hbm, "unit": "GB/s", "frac": split_gbs / hbm, "traffic": None,
                         "bytes_per_launch": w.kv_bytes()},
            "cpu_baseline": cpu,
            "e2e": {"value": w.kv_bytes() * world / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": q.numel() * q.element_size(),
                    "d2h_bytes_per_step": o.numel() * o.element_size() + lse.numel() * 4,
                    "ms_per_step": e2e_ms},
            "gpu_launches": gpu_launches,
            "clocks": clocks,
            "peak_source": f"{peak_src} hbm_gbs",
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


SIDE_WORKLOADS = ("tiny", "encoder", "gpt", "very_long")


def algorithmic_bytes(w):
    """(forward, backward) algorithmic HBM bytes of one step: the forward
    reads Q, K, V and writes O and LSE; the backward reads Q, K, V, O, dO,
    LSE and writes dQ, dK, dV (plus D, written and read back)."""
    T = w.B * w.N * w.H * w.d
    rows = w.B * w.H * w.N
    return 4 * T * 2 + 4 * rows, 8 * T * 2 + 2 * 4 * rows


def measure_device_only(attn, w, dev, warmup=3, target_ms=300.0):
    """fwd+bwd of workload w with inputs resident in HBM (drawn on the
    device from a seeded generator, N(0,1), Q and K times the workload's
    multiplier), timed by CUDA events on the launch stream and, in a second
    pass of the same steps, per kernel by the library's own events.  Used for
    the workloads besides the headline
    one, so that the whole N range of the metric is on one record."""
    import torch
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float16
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    shape = (w.B, w.N, w.H, w.d)
    q, k, v, do = (torch.randn(shape, generator=g, device=dev, dtype=torch.float32).to(dt)
                   for _ in range(4))
    if w.qk_mult != 1:
        q.mul_(w.qk_mult)
        k.mul_(w.qk_mult)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    ws = attn.workspace(w.B, w.H, w.N, w.d, dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        attn.check(attn.attn_fwd(q, k, v, o, lse, w.B, w.H, w.N, w.d, w.scale, w.causal, w.dtype,
                                 stream))
        attn.check(attn.attn_bwd(q, k, v, o, lse, do, dq, dk, dv, w.B, w.H, w.N, w.d, w.scale,
                                 w.causal, w.dtype, ws, ws.numel(), stream))

    for _ in range(warmup):
        step()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    steps = int(max(3, min(200, target_ms / max(e0.elapsed_time(e1), 1e-3))))
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    attn.check(attn.attn_status(stream))
    step_ms = e0.elapsed_time(e1) / steps
    # per-kernel durations from a second pass with the library's events
    # (kept out of the timed pass: they end the launches' programmatic overlap)
    attn.check(attn.attn_profile_begin())
    for _ in range(steps):
        step()
    torch.cuda.synchronize(dev)
    prof = attn.attn_profile_end()
    attn.check(attn.attn_status(stream))
    avg = {nm: (tot / n if n else None) for nm, (n, tot) in prof.items()}
    fwd_ms = avg["attn_fwd"]
    bwd_ms = sum(avg[nm] or 0.0 for nm in ("attn_bwd_pre", "attn_bwd_main", "attn_dq_post"))
    ffwd, fbwd = w.flops_fwd(), w.flops_bwd()
    fwd_bytes, bwd_bytes = algorithmic_bytes(w)
    return {
        "config": f"B={w.B} H={w.H} N={w.N} d={w.d} {w.dtype} "
                  f"{'causal' if w.causal else 'non-causal'}",
        "steps": steps, "ms_per_step": step_ms,
        "tflops": (ffwd + fbwd) / (step_ms * 1e-3) / 1e12,
        "fwd_tflops": ffwd / (fwd_ms * 1e-3) / 1e12,
        "bwd_tflops": fbwd / (bwd_ms * 1e-3) / 1e12,
        "bwd_main_tflops": fbwd / (avg["attn_bwd_main"] * 1e-3) / 1e12,
        "hbm_gbs": (fwd_bytes + bwd_bytes) / (step_ms * 1e-3) / 1e9,
        "fwd_hbm_gbs": fwd_bytes / (fwd_ms * 1e-3) / 1e9,
        "bwd_hbm_gbs": bwd_bytes / (bwd_ms * 1e-3) / 1e9,
        "kernel_ms": avg,
    }


def context_parallel_main(args, w):
    """Sequence parallelism's block kernels on one GPU: every rank's zigzag
    ring schedule over R ranks (attn_fwd_acc per block, then attn_bwd_acc per
    block in the ring's step order, then attn_cast_acc), run in one process
    with every shard resident (the exchange between GPUs is not timed: there
    is one GPU).  Same FLOP count as the plain workload; the plain kernels
    are timed in the same run for comparison."""
    import torch
    from exact_tiled_attention_22_gb300 import build
    build.build()
    from exact_tiled_attention_22_gb300 import attn
    from exact_tiled_attention_22_gb300 import context_parallel as cpm
    R = args.context_parallel
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if w.N % (2 * R):
        raise SystemExit(f"N = {w.N} is not a multiple of 2 x {R}")
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float16
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    full = [torch.randn((w.B, w.N, w.H, w.d), generator=g, device=dev, dtype=torch.float32).to(dt)
            for _ in range(4)]
    C = w.N // (2 * R)
    qs, ks, vs, dos = ([cpm.shard(t, R, r) for r in range(R)] for t in full)
    plans = [cpm.ring_plan(R, r, w.causal) for r in range(R)]
    os_ = [torch.empty_like(x) for x in qs]
    oacc = [torch.empty(x.shape, dtype=torch.float32, device=dev) for x in qs]
    lses = [torch.empty((2, w.B, w.H, C), dtype=torch.float32, device=dev) for _ in range(R)]
    dqs = [torch.empty_like(x) for x in qs]
    accs = [torch.empty((2,) + tuple(x.shape), dtype=torch.float32, device=dev) for x in ks]
    dks = [torch.empty_like(x) for x in ks]
    dvs = [torch.empty_like(x) for x in ks]
    wss = [[attn.workspace(w.B, w.H, C, w.d, dev) for _ in range(2)] for _ in range(R)]
    stream = torch.cuda.current_stream(dev)
    launches = [0]

    def step():
        for r in range(R):
            for st in plans[r]:
                for b in st.blocks:
                    attn.check(attn.attn_fwd_acc(qs[r][b.q_local], ks[st.src][b.kv_local], vs[st.src][b.kv_local],
                                                 oacc[r][b.q_local], lses[r][b.q_local], os_[r][b.q_local],
                                                 w.B, w.H, C, w.d, w.scale, b.causal, b.q_flags, w.dtype, stream))
                    launches[0] += 1
        for s_ in range(R):
            for r in range(R):
                st = plans[r][s_]
                for b in st.blocks:
                    qi, ki = b.q_local, b.kv_local
                    ws = wss[r][qi]
                    attn.check(attn.attn_bwd_acc(qs[r][qi], ks[st.src][ki], vs[st.src][ki], os_[r][qi],
                                                 lses[r][qi], dos[r][qi], dqs[r][qi], accs[st.src][0, ki],
                                                 accs[st.src][1, ki], w.B, w.H, C, w.d, w.scale, b.causal,
                                                 b.q_flags, b.kv_flags, w.dtype, ws, ws.numel(), stream))
                    launches[0] += 1 + (1 if b.q_flags & cpm.ACC_FIRST else 0) + (1 if b.q_flags & cpm.ACC_LAST else 0)
        for r in range(R):
            for c in range(2):
                for src, dst in ((accs[r][0, c], dks[r][c]), (accs[r][1, c], dvs[r][c])):
                    attn.check(attn.attn_cast_acc(src, dst, src.numel(), 1.0, w.dtype, stream))
                    launches[0] += 1

    for _ in range(args.warmup):
        step()
    attn.check(attn.attn_status(stream))
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(smi_id(0), gpu_uuid(dev))
    sampler.start()
    launches[0] = 0
    sampler.begin()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    sampler.end()
    clocks = sampler.stop()
    attn.check(attn.attn_status(stream))
    ms = e0.elapsed_time(e1) / args.steps
    plain = measure_device_only(attn, w, dev)
    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    value = (w.flops_fwd() + w.flops_bwd()) / (ms * 1e-3) / 1e12
    line = {
        "metric": "sequence-parallel block kernels on one GPU, fwd+bwd TFLOP/s", "value": value,
        "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": None, "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic",
        "config": dict(config_dict(w, args), context_parallel_ranks=R, chunk=C,
                       exchange="none timed: one GPU, every shard resident"),
        "pct_of_peak": 100.0 * value / peak, "peak_tflops": peak,
        "peak_source": peak_label(peak_src, w.dtype),
        "plain_same_run": {"tflops": plain["tflops"], "ms_per_step": plain["ms_per_step"]},
        "gpu_launches": launches[0], "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="long")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=30,
                    help="steps of the end-to-end pipeline in its timed region (its fill and "
                         "drain, one input and one output copy, are spread over them)")
    ap.add_argument("--alibi", action="store_true",
                    help="time the ALiBi variants (slopes 2^(-8(h+1)/H)); not the headline")
    ap.add_argument("--block-mask", default=None, metavar="PATTERN",
                    help="time the block-sparse variants with a 128 x 128 block mask: "
                         "'local_global:W' (band of W blocks plus the first block row and "
                         "column) or 'random:P' (each block kept with probability P); "
                         "FLOPs count only the scores the mask keeps; not the headline")
    ap.add_argument("--no-side", action="store_true",
                    help="skip the device-only measurement of the other fwd+bwd workloads "
                         "that the default long-workload run adds under 'workloads'")
    ap.add_argument("--all", action="store_true",
                    help="one full JSON line per fwd+bwd workload (tiny, encoder, gpt, long, "
                         "very_long), each from its own run of this script")
    ap.add_argument("--context-parallel", type=int, default=0, metavar="R",
                    help="time the sequence-parallel block kernels of an R-rank zigzag ring on "
                         "one GPU (every shard resident, no exchange); not the headline")
    ap.add_argument("--dropout", type=float, default=0.0, metavar="P",
                    help="time the dropout variants with probability P (seed 2024, a new "
                         "offset every step); same FLOP count; not the headline")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    from exact_tiled_attention_22_gb300.inputs import DECODE_WORKLOADS, WORKLOADS
    if args.all:
        passthrough = [a for a in sys.argv[1:] if a != "--all"]
        passthrough = [a for i, a in enumerate(passthrough)
                       if a != "--workload" and (i == 0 or passthrough[i - 1] != "--workload")
                       and not a.startswith("--workload=")]
        rc = 0
        for name in ("tiny", "encoder", "gpt", "long", "very_long"):
            r = subprocess.run([sys.executable, os.path.abspath(__file__), "--workload", name,
                                "--no-side"] + passthrough)
            rc = rc or r.returncode
        return rc
    if args.workload in DECODE_WORKLOADS:
        return decode_main(args, DECODE_WORKLOADS[args.workload])
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        return reference_arm(args, w)
    if args.context_parallel:
        return context_parallel_main(args, w)

    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    from exact_tiled_attention_22_gb300 import build
    build.build()
    from exact_tiled_attention_22_gb300 import attn
    from exact_tiled_attention_22_gb300.inputs import workload_inputs

    B, H, N, d = w.B, w.H, w.N, w.d
    x = workload_inputs(w)
    near = gpu_local_cpus(gpu_uuid(dev) or "")
    with on_cpus(near):
        host = {n: t.pin_memory() for n, t in x.items()}
    q, k, v, do = (host[n].to(dev) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    ws = attn.workspace(B, H, N, d, dev)
    stream = torch.cuda.current_stream(dev)
    slopes = (torch.tensor([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)], dtype=torch.float32,
                           device=dev) if args.alibi else None)
    mask_host, bmask, kept = None, None, None
    if args.block_mask:
        pattern, _, par = args.block_mask.partition(":")
        from exact_tiled_attention_22_gb300.inputs import make_block_mask
        if pattern == "local_global":
            mask_host = make_block_mask(H, N, pattern, width=int(par or 1))
        else:
            mask_host = make_block_mask(H, N, pattern, density=float(par or 0.5), seed=w.seed)
        kept = kept_pairs(mask_host, N, w.causal)
        mask_host = mask_host.pin_memory()
        bmask = mask_host.to(dev)

    n_step = [0]
    main_bufs = dict(q=q, k=k, v=v, do=do, o=o, lse=lse, dq=dq, dk=dk, dv=dv, bmask=bmask)

    def run_step(bf, strm):
        """One fwd+bwd step on the device buffers bf, launched on strm."""
        off = n_step[0]
        n_step[0] += 1
        attn.check(attn.attn_fwd_ex(bf["q"], bf["k"], bf["v"], bf["o"], bf["lse"], B, H, N, d,
                                    w.scale, w.causal, slopes, bf["bmask"], args.dropout, 2024,
                                    off, w.dtype, strm))
        attn.check(attn.attn_bwd_ex(bf["q"], bf["k"], bf["v"], bf["o"], bf["lse"], bf["do"],
                                    bf["dq"], bf["dk"], bf["dv"], B, H, N, d, w.scale, w.causal,
                                    slopes, bf["bmask"], args.dropout, 2024, off, w.dtype, ws,
                                    ws.numel(), strm))

    def step():
        run_step(main_bufs, stream)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        step()
    attn.check(attn.attn_status(stream))
    torch.cuda.synchronize(dev)

    sampler = ClockSampler(smi_id(local), gpu_uuid(dev)) if rank == 0 else None
    if sampler:
        sampler.start()
    barrier()
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.begin()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.end()
    barrier()
    clocks = sampler.stop() if sampler else None
    attn.check(attn.attn_status(stream))
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    # Per-kernel durations: the same K steps again, each launch bracketed by
    # the library's own CUDA events on the launch stream.  (Not in the timed
    # region above: an event between two launches ends the programmatic
    # overlap of one kernel's launch with the previous kernel's tail.)
    attn.check(attn.attn_profile_begin())
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize(dev)
    prof = attn.attn_profile_end()
    attn.check(attn.attn_status(stream))
    gpu_launches = sum(n for n, _ in prof.values())

    # ---- end to end through the C ABI with pinned host buffers ----
    # A two-deep pipeline, as a training input pipeline runs it: while the
    # kernels of step i run on the compute stream, step i+1's inputs are
    # copied in on one copy stream and step i's results are copied out on
    # another as soon as they exist.  Device buffers and pinned host result
    # buffers are double-buffered; every step's inputs and results cross the
    # host link inside the timed region.
    in_names, out_names = ("q", "k", "v", "do"), ("o", "lse", "dq", "dk", "dv")
    bufs = [main_bufs, {n: torch.empty_like(t) for n, t in main_bufs.items() if t is not None}]
    bufs[1].setdefault("bmask", None)
    with on_cpus(near):
        out_host = [{n: torch.empty(bufs[0][n].shape, dtype=bufs[0][n].dtype).pin_memory()
                     for n in out_names} for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = {key: [torch.cuda.Event() for _ in range(2)] for key in ("in", "done", "out")}

    def copy_in(b, after_step_used_it):
        with torch.cuda.stream(s_in):
            if after_step_used_it:
                s_in.wait_event(ev["done"][b])  # the step that read these inputs is over
            for n in in_names:
                bufs[b][n].copy_(host[n], non_blocking=True)
            if mask_host is not None:
                bufs[b]["bmask"].copy_(mask_host, non_blocking=True)
            ev["in"][b].record(s_in)

    def e2e_run(n_steps, start_event=None):
        if start_event is not None:
            s_in.wait_event(start_event)
        copy_in(0, False)
        for i in range(n_steps):
            b, nb = i % 2, (i + 1) % 2
            if i + 1 < n_steps:
                copy_in(nb, i >= 1)
            stream.wait_event(ev["in"][b])
            if i >= 2:
                stream.wait_event(ev["out"][b])  # step i-2's results have left
            run_step(bufs[b], stream)
            ev["done"][b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev["done"][b])
                for n in out_names:
                    out_host[b][n].copy_(bufs[b][n], non_blocking=True)
                ev["out"][b].record(s_out)
        stream.wait_event(ev["out"][(n_steps - 1) % 2])

    e2e_run(2)
    torch.cuda.synchronize(dev)
    barrier()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    e2e_run(args.e2e_steps, start_event=f0)
    f1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    e2e_ms = max_over_ranks(f0.elapsed_time(f1), world, dev)
    attn.check(attn.attn_status(stream))
    h2d = sum(host[n].numel() * host[n].element_size() for n in in_names)
    if mask_host is not None:
        h2d += mask_host.numel()
    d2h = sum(t.numel() * t.element_size() for t in out_host[0].values())

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    ffwd, fbwd = w.flops_fwd(), w.flops_bwd()
    if kept is not None:  # scores the mask keeps: 4 d flops each forward, 2.5x that backward
        ffwd = 4.0 * d * B * kept
        fbwd = 2.5 * ffwd
    step_ms = ms / args.steps
    value = aggregate_tflops(ffwd + fbwd, world, step_ms)
    e2e_value = aggregate_tflops(ffwd + fbwd, world, e2e_ms / args.e2e_steps)
    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])

    avg = {name: (tot / n if n else None) for name, (n, tot) in prof.items()}
    bwd_ms = sum(a for nm, a in avg.items() if nm != "attn_fwd" and a)
    # achieved HBM bandwidth of the algorithmic bytes, against the measured
    # copy bandwidth (the short shapes are bound by neither pipe)
    fb, bb = algorithmic_bytes(w)
    hbm_peak = float(peaks["hbm_gbs"])
    step_gbs = (fb + bb) * world / (step_ms * 1e-3) / 1e9
    hbm_line = {"step_gbs": step_gbs, "fwd_gbs": fb / (avg["attn_fwd"] * 1e-3) / 1e9,
                "bwd_gbs": bb / (bwd_ms * 1e-3) / 1e9, "bytes_per_step": fb + bb,
                "peak_gbs": hbm_peak, "frac": step_gbs / (hbm_peak * world)}
    # the backward's HBM-bound helpers against the measured copy bandwidth:
    # pre reads O, dO and LSE, writes -LSE log2 e and D and clears the fp32 dQ
    # accumulator (rows padded to 128); post reads the accumulator's N rows
    # and writes dQ
    T = B * N * H * d
    rows, rows_pad = B * H * N, B * H * ((N + 127) // 128 * 128)
    pre_bytes = 2 * T * 2 + 4 * rows + 2 * 4 * rows_pad + 4 * rows_pad * d
    post_bytes = T * 4 + T * 2
    aux = {}
    for nm, nb in (("attn_bwd_pre", pre_bytes), ("attn_dq_post", post_bytes)):
        if avg.get(nm):
            gbs = nb / (avg[nm] * 1e-3) / 1e9
            aux[nm] = {"bytes": nb, "gbs": gbs, "frac": gbs / hbm_peak}
    main_ms = avg["attn_bwd_main"]
    achieved = fbwd / (main_ms * 1e-3) / 1e12
    traffic = (bwd_main_traffic(w.name) if not (args.block_mask or args.alibi or args.dropout)
               else None)

    cpu = None
    if world == 1 and not args.no_cpu_baseline and not args.block_mask and not args.dropout:
        cv, cdt, cn, cth, cheads = oracle_sample(w, 15.0)
        cpu = {"value": cv, "unit": UNIT, "cores": cth, "kind": "oracle",
               "sample": sample_text(w, cn, cheads, cdt)}

    side = None
    if (world == 1 and not args.no_side and w.name == "long" and not args.block_mask
            and not args.alibi and not args.dropout):
        side = {}
        for name in SIDE_WORKLOADS:
            r = measure_device_only(attn, WORKLOADS[name], dev)
            r["pct_of_peak"] = 100.0 * r["tflops"] / peak
            side[name] = r

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": config_dict(w, args, None if kept is None else (4.0 * d * B * kept) / w.flops_fwd()),
        "pct_of_peak": 100.0 * value / (peak * world),
        "peak_tflops": peak, "peak_source": peak_label(peak_src, w.dtype),
        "fwd_tflops": ffwd / (avg["attn_fwd"] * 1e-3) / 1e12,
        "bwd_tflops": fbwd / (bwd_ms * 1e-3) / 1e12,
        "kernel_ms": {nm: a for nm, a in avg.items()},
        "hbm": hbm_line,
        "hbm_bound_kernels": aux,
        "roofline": {"kernel": "attn_bwd_main", "bound": "tensor", "achieved": achieved,
                     "peak": peak, "unit": UNIT, "frac": achieved / peak, "traffic": traffic,
                     "flops_per_launch": fbwd},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / args.e2e_steps,
                "host_buffers_from_gpu_local_cpus": bool(near)},
        "gpu_launches": gpu_launches,
        "clocks": clocks,
        "workloads": side,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
