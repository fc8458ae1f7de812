#!/usr/bin/env python
"""Benchmark of exact attention on GB300: one step = forward + backward of causal
bf16 attention, B=2 H=32 N=8192 d=128, through the library's C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line.  ``value`` is attention TFLOP/s over the whole step
(forward 4 N^2 d per head halved for causal, backward 2.5x forward), inputs
resident in device memory, L2 flushed between steps (untimed), CUDA events on the
launching stream.  ``--impl reference`` times the fp64 CPU oracle on a bounded
sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention TFLOPS (fwd, fwd+bwd) bf16 N=8k d=128 causal; % of GB300 tensor peak"
WORKLOAD_ID = 3      # B=2 H=32 N=8192 d=128 causal, bf16
CAUSAL = True
L2_FLUSH_BYTES = 256 << 20
CPU_SAMPLE_ROWS = 256   # query rows per head timed on the host for cpu_baseline
E2E_CHUNK_HEADS = 4     # heads per chunk of the host-buffer pipeline (e2e)
REF_STEP_ROWS = 32      # query rows per head per step of the reference arm


class L2Flush:
    """Evicts the inputs from L2 between timed calls (untimed): a 256 MiB write, larger
    than the 129 MB L2, then a 256 MiB read, so that L2 is left holding clean lines.  The
    write alone leaves about an L2's worth of dirty lines, whose write-back to DRAM the
    next timed kernel would pay for (~14 us of a 105 us decoding call)."""

    def __init__(self, dev):
        import torch
        self.torch = torch
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.torch.amax(self.r, dim=0, out=self.sink)


L2_NOTE = "L2 flushed between timed calls (256 MiB write, then a 256 MiB read: no dirty lines left)"


# DRAM bytes (read + write) per call of the bench shape, from one ncu capture of
# dram__bytes_read.sum + dram__bytes_write.sum over every launch of the attention kernels
# (`ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum --clock-control none
# -k "regex:fwd_kernel|bwd_" python bench.py --shape 1,32,8192,128 --steps 1 --warmup 3
# --no-cpu-baseline --no-e2e`: half the heads of the bench shape, scaled by 2).  A figure is reported only while the kernel sources still hash to the value
# they had when the counters were taken; after any change it reads as null until the
# capture is repeated.
TRAFFIC = {
    "bwd": (2017.8e6, ('fa_bwd.cu', 'fa_api.cu', 'ptx.cuh', 'fa_internal.h'), "0cf0e239c7bbda6a"),
    "bwd_det": (1660.6e6, ('fa_bwd.cu', 'fa_api.cu', 'ptx.cuh', 'fa_internal.h'), "0cf0e239c7bbda6a"),
    "fwd": (491.0e6, ('fa_fwd.cu', 'ptx.cuh', 'fa_internal.h'), "77d64738ea74f26c"),
}


def measured_traffic(kernel, shape):
    import hashlib
    entry = TRAFFIC.get(kernel)
    if entry is None or shape is not None:
        return None
    nbytes, files, want = entry
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "exact_attention_tmem_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return nbytes if h.hexdigest()[:16] == want else None


def flops_fwd_rows(rows, d, heads, causal=True, n=None):
    """Forward FLOPs of the listed query rows: 4 d (visible keys) per row."""
    if causal:
        keys = sum(int(r) + 1 for r in rows)
    else:
        keys = len(rows) * n
    return 4.0 * d * keys * heads


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), \
            float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, 1700.0, 6800.0, "fallback"


class NvmlPoller:
    """SM clock and clock-event reasons read through NVML (read-only queries) every
    few milliseconds from a host thread, so that even a timed region of a few
    milliseconds holds several samples.  The device is matched by UUID."""
    SM = 1                           # NVML_CLOCK_SM
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid, index, period_s=0.002):
        import ctypes
        import threading
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        rc = 1
        if uuid:
            rc = self.lib.nvmlDeviceGetHandleByUUID(("GPU-" + uuid).encode(), ctypes.byref(self.h))
        if rc != 0:
            rc = self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h))
        if rc != 0:
            raise OSError("no NVML handle for the device")
        self.reason_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        self.max_mhz = float(mx.value) if self.lib.nvmlDeviceGetMaxClockInfo(
            self.h, self.SM, ctypes.byref(mx)) == 0 else None
        self.period = period_s
        self.samples, self.reasons = [], set()
        self.stop_ev = threading.Event()
        self.thread = threading.Thread(target=self._run, daemon=True)

    def _run(self):
        ct = self.ct
        mhz, bits = ct.c_uint(), ct.c_ulonglong()
        while not self.stop_ev.is_set():
            if self.lib.nvmlDeviceGetClockInfo(self.h, self.SM, ct.byref(mhz)) == 0:
                self.samples.append(float(mhz.value))
            if self.reason_fn(self.h, ct.byref(bits)) == 0:
                for bit, name in self.REASONS.items():
                    if bits.value & bit:
                        self.reasons.add(name)
            self.stop_ev.wait(self.period)

    def start(self):
        self.thread.start()

    def stop(self):
        self.stop_ev.set()
        self.thread.join(timeout=5)
        self.lib.nvmlShutdown()

    def summary(self):
        if not self.samples:
            return None
        return {"sm_mhz": statistics.median(self.samples),
                "sm_max_mhz": self.max_mhz if self.max_mhz else max(self.samples),
                "samples": len(self.samples), "source": "nvml", "reasons": sorted(self.reasons)}


class ClockSampler:
    """Clocks and throttle reasons of the bench's GPU during the timed region: NVML
    polled from a host thread, else nvidia-smi sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None
        self.nvml = None

    def _uuid(self):
        try:
            import torch
            return str(torch.cuda.get_device_properties(self.index).uuid)
        except Exception:
            return None

    def __enter__(self):
        try:
            self.nvml = NvmlPoller(self._uuid(), self.index)
            self.nvml.start()
            return self
        except (OSError, AttributeError):
            self.nvml = None
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            dev_id = self._uuid()
            dev_id = ("GPU-" + dev_id) if dev_id else str(self.index)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={dev_id}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.nvml is not None:
            self.nvml.stop()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.nvml is not None:
            return self.nvml.summary()
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return None
        rows = list(csv.reader(io.StringIO(open(self.path).read())))
        os.unlink(self.path)
        sm, mx, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names[1:], r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "source": "nvidia-smi", "reasons": sorted(reasons)}


def dist_setup(backend):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend=backend)
    return world, rank, local


def max_over_ranks(value, device="cpu"):
    """The slowest rank's value (the job is only as fast as its slowest replica)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world, steps, flops_per_rank_step, total_ms):
    """Whole-job throughput: every rank runs its own replica of the step."""
    return world * steps * flops_per_rank_step / (total_ms * 1e-3) / 1e12


def cpu_oracle_sample(q, k, v, do, d, rows):
    """Time the fp64 oracle (forward + backward) on the listed query rows of every head."""
    import oracle
    from exact_attention_tmem_gb300 import inputs
    q64, k64, v64, do64 = (inputs.as_f64(t) for t in (q, k, v, do))
    scale = 1.0 / math.sqrt(d)
    heads = q.shape[0] * q.shape[1]
    t0 = time.perf_counter()
    oracle.attention_fwd_rows(q64, k64, v64, scale, CAUSAL, rows)
    oracle.attention_bwd_rows(q64, k64, v64, do64, scale, CAUSAL, rows)
    dt = time.perf_counter() - t0
    fl = 3.5 * flops_fwd_rows(rows, d, heads, CAUSAL)
    return fl / dt / 1e12, dt, oracle.num_threads()


def run_reference(args, world, rank):
    """The reference arm: the fp64 CPU oracle, as it stands, on sampled rows."""
    if rank != 0:
        return
    from exact_attention_tmem_gb300 import inputs
    w = inputs.WORKLOADS[WORKLOAD_ID]
    q, k, v, do = inputs.workload_inputs(WORKLOAD_ID, with_grad_out=True)
    times, cores, fl = [], 1, 0.0
    for step in range(args.warmup + args.steps):
        rows = inputs.sample_rows(w.N, REF_STEP_ROWS, seed=100 + step)
        tf, dt, cores = cpu_oracle_sample(q, k, v, do, w.d, rows)
        if step >= args.warmup:
            times.append(dt)
            fl += 3.5 * flops_fwd_rows(rows, w.d, w.B * w.H, CAUSAL)
    value = fl / sum(times) / 1e12
    sample = (f"{REF_STEP_ROWS} seeded query rows of each of the {w.B * w.H} heads per step "
              "(forward + backward of those rows, fp64)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_dict(w),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


FP8_METRIC = "attention TFLOPS (fwd), fp8 e4m3 with incoherent processing, N=8k d=128 causal (fa_fwd_fp8)"
FP8_NOMINAL_RATIO = 2.0   # dense fp8 / dense bf16 tensor rate (4.5 / 2.25 PFLOP/s nominal)


def run_fp8(args, world, rank, local):
    """FP8 forward on workload 3's shape: Q and K rotated and quantized, V quantized and
    transposed, outside the timed region (a model would keep them in fp8); the timed call
    is fa_fwd_fp8.  The peak is the measured bf16 peak times the nominal fp8/bf16 ratio."""
    import torch
    import numpy as np
    import exact_attention_tmem_gb300 as fa
    from exact_attention_tmem_gb300 import inputs

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fa.build()
    w = inputs.WORKLOADS[WORKLOAD_ID]
    B, H, N, d = args.shape if args.shape else (w.B, w.H, w.N, w.d)
    if args.shape:
        q_h, k_h, v_h = inputs.random_inputs(B, H, N, d, seed=WORKLOAD_ID)
    else:
        q_h, k_h, v_h = inputs.workload_inputs(WORKLOAD_ID)
    q, k, v = (t.to(dev) for t in (q_h, k_h, v_h))
    signs = torch.from_numpy(np.random.default_rng(41).choice([-1.0, 1.0], size=d).astype(np.float32)).to(dev)
    q8, dq = fa.quantize_qk_fp8(q, signs)
    k8, dk = fa.quantize_qk_fp8(k, signs)
    vt8, dv = fa.quantize_v_fp8(v)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)

    def call():
        fa.fwd_fp8(q8, k8, vt8, dq, dk, dv, causal=CAUSAL, out=o, lse=lse)

    for _ in range(args.warmup):
        call()
        flush()
    torch.cuda.synchronize(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            flush()
            ev[i][0].record(stream)
            call()
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    status = fa.device_status()
    total_ms = max_over_ranks(sum(e[0].elapsed_time(e[1]) for e in ev), dev)
    flops = 4.0 * N * N * d * B * H / (2 if CAUSAL else 1)
    value = job_tflops(world, args.steps, flops, total_ms)
    e2e = None
    if not args.no_e2e:
        # the codes come from pinned host memory, O and L go back
        hq, hk, hv = (t.cpu().pin_memory() for t in (q8, k8, vt8))
        ho = torch.empty(tuple(o.shape), dtype=torch.bfloat16).pin_memory()
        hl = torch.empty(tuple(lse.shape), dtype=torch.float32).pin_memory()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            for dst, src in ((q8, hq), (k8, hk), (vt8, hv)):
                dst.copy_(src, non_blocking=True)
            call()
            ho.copy_(o, non_blocking=True)
            hl.copy_(lse, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / args.steps
        e2e = {"value": world * flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": sum(t.numel() for t in (hq, hk, hv)),
               "d2h_bytes_per_step": ho.numel() * 2 + hl.numel() * 4, "ms_per_step": ms}
    if rank != 0:
        return
    peak_burst, _, _, peak_src = peaks()
    peak8 = peak_burst * FP8_NOMINAL_RATIO
    tf = value / world
    line = {
        "metric": FP8_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 (fp32 accumulate, bf16 out)", "data": "synthetic",
        "config": {"workload": f"fwd fp8 causal B={B} H={H} N={N} d={d}", "B": B, "H": H, "N": N, "d": d,
                   "causal": CAUSAL, "scale": "1/sqrt(d)", "inputs": "workload 3's bf16 inputs, Q and K rotated by "
                   "diag(s) H / sqrt(d) (signs seed 41), e4m3 codes with one scale per head",
                   "l2": "inputs > L2; " + L2_NOTE,
                   "parallelism": "one independent replica per GPU"},
        "roofline": {"bound": "tensor", "kernel": "fwd_fp8_kernel (CUDA events around the C-ABI call)",
                     "achieved": tf, "peak": peak8, "unit": "TFLOP/s", "frac": tf / peak8, "traffic": None,
                     "peak_source": f"{peak_src} bf16 burst x {FP8_NOMINAL_RATIO:g} (nominal fp8/bf16 ratio)"},
        "e2e": e2e, "gpu_launches": args.steps, "device_status": status, "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


DECODE_METRIC = "decode K/V read bandwidth, bf16, one query row per head (fa_decode)"
DECODE_SHAPE = (8, 32, 32, 32768, 128)     # B, H, Hkv, Nk, d


def run_decode(args, world, rank, local):
    """Decoding: one query row per head against Nk keys (split-key kernel + merge).
    The metric is the compulsory K/V (+ q, o) bytes per call over the call's time,
    against the measured HBM copy bandwidth: the kernel streams K and V once."""
    import torch
    import exact_attention_tmem_gb300 as fa
    from exact_attention_tmem_gb300 import inputs

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fa.build()
    B, H, Hkv, Nk, d = args.decode_shape or DECODE_SHAPE
    scale = 1.0 / math.sqrt(d)
    q_h = inputs.normal((B, H, d), 21001)
    k_h = inputs.normal((B, Hkv, Nk, d), 21002)
    v_h = inputs.normal((B, Hkv, Nk, d), 21003)
    q, k, v = (t.to(dev) for t in (q_h, k_h, v_h))
    o = torch.empty_like(q)
    lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    ws = torch.empty(fa.decode_workspace_size(B, H, Hkv, Nk, d), dtype=torch.uint8, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    nbytes = 2 * B * Hkv * Nk * d * 2 + 2 * B * H * d * 2 + B * H * 4

    def call():
        fa.decode(q, k, v, scale=scale, out=o, lse=lse, workspace=ws)

    for _ in range(args.warmup):
        call()
        flush()
    torch.cuda.synchronize(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            flush()
            ev[i][0].record(stream)
            call()
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    status = fa.device_status()
    t = [e[0].elapsed_time(e[1]) for e in ev]
    total_ms = max_over_ranks(sum(t), dev)
    gbs = world * nbytes * args.steps / (total_ms * 1e-3) / 1e9
    # end to end: the query rows come from pinned host memory, o and lse go back; the
    # K/V cache stays resident on the device as a decoder's cache would
    e2e = None
    if not args.no_e2e:
        hq = q_h.pin_memory()
        ho = torch.empty_like(q_h).pin_memory()
        hl = torch.empty((B, H), dtype=torch.float32).pin_memory()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            q.copy_(hq, non_blocking=True)
            call()
            ho.copy_(o, non_blocking=True)
            hl.copy_(lse, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / args.steps
        e2e = {"value": world * nbytes / (ms * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": hq.numel() * 2, "d2h_bytes_per_step": ho.numel() * 2 + hl.numel() * 4,
               "ms_per_step": ms}
    if rank != 0:
        return
    _, _, hbm, peak_src = peaks()
    line = {
        "metric": DECODE_METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"decode B={B} H={H} Hkv={Hkv} Nk={Nk} d={d}", "B": B, "H": H, "Hkv": Hkv,
                   "Nk": Nk, "d": d, "scale": "1/sqrt(d)", "inputs": "iid N(0,1) rounded to bf16, seeds 21001-21003",
                   "l2": "K/V larger than L2; " + L2_NOTE,
                   "parallelism": "one independent replica per GPU"},
        "roofline": {"bound": "hbm", "kernel": "decode_split_kernel + decode_combine_kernel (CUDA events around "
                     "the C-ABI call)", "achieved": gbs / world, "peak": hbm, "unit": "GB/s",
                     "frac": gbs / world / hbm, "traffic": None,
                     "algorithmic_bytes_per_call": nbytes, "peak_source": f"{peak_src} HBM copy"},
        "e2e": e2e, "gpu_launches": 2 * args.steps, "device_status": status, "clocks": clk.summary(),
    }
    if world == 1 and not args.no_cpu_baseline:
        from oracle import decode as odec
        heads = min(B * H, 4)
        f = inputs.as_f64
        qs, ks, vs = f(q_h[0, :heads])[None], f(k_h[0]), f(v_h[0])
        kv = [h // (H // Hkv) for h in range(heads)]
        t0 = time.perf_counter()
        for h in range(heads):
            odec.attention_decode(qs[:, h:h + 1], ks[None, kv[h]:kv[h] + 1], vs[None, kv[h]:kv[h] + 1], scale)
        dt = time.perf_counter() - t0
        sample_bytes = heads * 2 * Nk * d * 2
        line["cpu_baseline"] = {"value": sample_bytes / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                "sample": f"{heads} query heads of batch 0 (numpy fp64), {dt:.2f} s"}
    print(json.dumps(line), flush=True)


def config_dict(w, shape=None, deterministic=False):
    B, H, N, d = shape if shape else (w.B, w.H, w.N, w.d)
    return {"workload": f"fwd+bwd causal bf16 B={B} H={H} N={N} d={d}",
            "B": B, "H": H, "N": N, "d": d, "causal": CAUSAL, "scale": "1/sqrt(d)",
            "backward": "deterministic (fa_bwd_deterministic)" if deterministic else "default (fa_bwd)",
            "inputs": "iid N(0,1) rounded to bf16, seeds 3001-3004",
            "l2": "inputs 512 MiB > L2; " + L2_NOTE,
            "parallelism": "one independent replica per GPU"}


def run_ours(args, world, rank, local):
    import torch
    import exact_attention_tmem_gb300 as fa
    from exact_attention_tmem_gb300 import inputs

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fa.build()
    w = inputs.WORKLOADS[WORKLOAD_ID]
    B, H, N, d = args.shape if args.shape else (w.B, w.H, w.N, w.d)
    scale = 1.0 / math.sqrt(d)
    if args.shape:
        q_h, k_h, v_h, do_h = inputs.random_inputs(B, H, N, d, seed=WORKLOAD_ID, with_grad_out=True)
    else:
        q_h, k_h, v_h, do_h = inputs.workload_inputs(WORKLOAD_ID, with_grad_out=True)
    q, k, v, do = (t.to(dev) for t in (q_h, k_h, v_h, do_h))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    det = bool(args.deterministic)
    ws_bytes = (fa.bwd_deterministic_workspace_size if det else fa.bwd_workspace_size)(B, H, N, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        fa.fwd(q, k, v, causal=CAUSAL, scale=scale, out=o, lse=lse)
        fa.bwd(q, k, v, o, lse, do, causal=CAUSAL, scale=scale, dq=dq, dk=dk, dv=dv, workspace=ws,
               deterministic=det)

    for _ in range(args.warmup):
        step()
        flush()
    torch.cuda.synchronize(dev)
    if fa.device_status() != 0:
        raise RuntimeError("device status reports a timed-out wait during warm-up")

    fwd_flops = 4.0 * N * N * d * B * H / (2 if CAUSAL else 1)
    bwd_flops = 2.5 * fwd_flops
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            flush()
            ev[i][0].record(stream)
            fa.fwd(q, k, v, causal=CAUSAL, scale=scale, out=o, lse=lse)
            ev[i][1].record(stream)
            fa.bwd(q, k, v, o, lse, do, causal=CAUSAL, scale=scale, dq=dq, dk=dk, dv=dv, workspace=ws,
                   deterministic=det)
            ev[i][2].record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    status = fa.device_status()
    t_fwd = [ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps)]
    t_bwd = [ev[i][1].elapsed_time(ev[i][2]) for i in range(args.steps)]
    t_step = [a + b for a, b in zip(t_fwd, t_bwd)]
    total_ms = max_over_ranks(sum(t_step), dev)
    value = job_tflops(world, args.steps, fwd_flops + bwd_flops, total_ms)
    fwd_tf = fwd_flops / (statistics.mean(t_fwd) * 1e-3) / 1e12
    bwd_tf = bwd_flops / (statistics.mean(t_bwd) * 1e-3) / 1e12

    # ---- end to end through the public API: pinned host inputs in, results back out
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, world, dev, stream, (q_h, k_h, v_h, do_h), CAUSAL, scale, fwd_flops + bwd_flops)
    if rank != 0:
        return
    peak_burst, peak_sust, hbm, peak_src = peaks()
    dominant = "bwd" if statistics.mean(t_bwd) >= statistics.mean(t_fwd) else "fwd"
    dom_tf = bwd_tf if dominant == "bwd" else fwd_tf
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_dict(w, args.shape, det),
        "fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf,
        "fwd_ms": statistics.mean(t_fwd), "bwd_ms": statistics.mean(t_bwd),
        "fwd_frac_of_peak": fwd_tf / peak_burst, "bwd_frac_of_peak": bwd_tf / peak_burst,
        "roofline": {"bound": "tensor", "kernel": f"{dominant} (CUDA events around the C-ABI call)",
                     "achieved": dom_tf, "peak": peak_burst, "unit": "TFLOP/s",
                     "frac": dom_tf / peak_burst,
                     "traffic": measured_traffic(dominant + ("_det" if det and dominant == "bwd" else ""),
                                                 args.shape),
                     "traffic_unit": "bytes per call (DRAM read + write, ncu)",
                     "peak_source": f"{peak_src} bf16 burst"},
        "e2e": e2e,
        "gpu_launches": 4 * args.steps,
        "device_status": status,
    }
    clocks = clk.summary()
    line["clocks"] = clocks
    if world == 1 and not args.no_cpu_baseline:
        rows = inputs.sample_rows(N, CPU_SAMPLE_ROWS, seed=7)
        tf, dt, cores = cpu_oracle_sample(q_h, k_h, v_h, do_h, d, rows)
        line["cpu_baseline"] = {
            "value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": (f"{len(rows)} seeded query rows of each of the {B * H} heads, forward + "
                       f"backward of those rows in fp64, {dt:.1f} s")}
    print(json.dumps(line), flush=True)


def run_e2e(args, world, dev, stream, host_in, causal, scale, flops):
    """The same step through the host-buffer entry point fa_fwd_bwd_host: pinned host
    inputs in, every output back in pinned host memory, the library overlapping the
    copies of one chunk of heads with the kernels of another; host-device copies are
    inside the timed region."""
    import torch
    import exact_attention_tmem_gb300 as fa
    q_h, k_h, v_h, do_h = host_in
    B, H, N, d = q_h.shape
    hq, hk, hv, hdo = (t.pin_memory() for t in (q_h, k_h, v_h, do_h))
    ho, hdq, hdk, hdv = (torch.empty_like(t).pin_memory() for t in (q_h, q_h, k_h, v_h))
    hlse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo))
    d2h = sum(t.numel() * t.element_size() for t in (ho, hlse, hdq, hdk, hdv))
    chunk = E2E_CHUNK_HEADS
    buf = torch.empty(fa.fwd_bwd_host_buffer_size(B, H, N, d, chunk), dtype=torch.uint8, device=dev)

    def e2e_step():
        fa.fwd_bwd_host(hq, hk, hv, hdo, causal=causal, scale=scale, o=ho, lse=hlse, dq=hdq, dk=hdk, dv=hdv,
                        buffer=buf, chunk_heads=chunk)

    e2e_steps = max(1, min(args.steps, 5))
    for _ in range(2):   # warm-up: first use of the pinned buffers and of the library's streams
        e2e_step()
    torch.cuda.synchronize(dev)
    # one event pair per step, back to back on the stream: the sum is the whole span
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps + 1)]
    ev[0].record(stream)
    for i in range(e2e_steps):
        e2e_step()
        ev[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    step_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(e2e_steps)]
    e2e_ms = max_over_ranks(sum(step_ms), dev) / e2e_steps
    return {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
            "step_ms": [round(t, 3) for t in step_ms],
            "path": f"fa_fwd_bwd_host, pinned host buffers, chunks of {chunk} heads"}


def run_link(args, world, rank, local):
    """Host-link bandwidth for the end-to-end step's bytes (pinned host memory): the step's
    inputs host->device alone, its outputs device->host alone, and both at once on two
    streams.  The last is the floor for ``e2e``: every byte has to cross the link."""
    import torch

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B, H, N, d = args.shape or (2, 32, 8192, 128)
    n_in = 4 * B * H * N * d * 2                   # q, k, v, dO (bf16)
    n_out = 4 * B * H * N * d * 2 + B * H * N * 4  # o, dq, dk, dv (bf16) and L (fp32)
    hin = torch.empty(n_in, dtype=torch.uint8).pin_memory()
    hout = torch.empty(n_out, dtype=torch.uint8).pin_memory()
    din = torch.empty(n_in, dtype=torch.uint8, device=dev)
    dout = torch.empty(n_out, dtype=torch.uint8, device=dev)
    cur = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def copies(up, down):
        s_in.wait_stream(cur)
        s_out.wait_stream(cur)
        if up:
            with torch.cuda.stream(s_in):
                din.copy_(hin, non_blocking=True)
        if down:
            with torch.cuda.stream(s_out):
                hout.copy_(dout, non_blocking=True)
        cur.wait_stream(s_in)
        cur.wait_stream(s_out)

    res = {}
    for name, up, down in (("h2d", True, False), ("d2h", False, True), ("both", True, True)):
        for _ in range(args.warmup):
            copies(up, down)
        torch.cuda.synchronize(dev)
        ts = []
        for _ in range(args.steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(cur)
            copies(up, down)
            e1.record(cur)
            torch.cuda.synchronize(dev)
            ts.append(e0.elapsed_time(e1))
        res[name] = statistics.median(ts)
    if rank != 0:
        return
    line = {
        "metric": "host link bandwidth, pinned host memory, the bench step's bytes", "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "config": {"workload": f"fwd+bwd B={B} H={H} N={N} d={d}: inputs in, outputs out",
                   "bytes_in": n_in, "bytes_out": n_out},
        "h2d_gbs": n_in / (res["h2d"] * 1e-3) / 1e9, "d2h_gbs": n_out / (res["d2h"] * 1e-3) / 1e9,
        "both_gbs": (n_in + n_out) / (res["both"] * 1e-3) / 1e9,
        "h2d_ms": res["h2d"], "d2h_ms": res["d2h"], "both_ms": res["both"],
        "e2e_floor_ms": res["both"],
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip timing the fp64 oracle on the host")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end (host buffers) measurement")
    ap.add_argument("--fp8", action="store_true",
                    help="time the FP8 forward (fa_fwd_fp8) on the same shape instead of the bf16 step")
    ap.add_argument("--decode", action="store_true",
                    help="time the decoding kernel (one query row per head) instead of the fwd+bwd step")
    ap.add_argument("--decode-shape", type=lambda x: tuple(int(v) for v in x.split(",")), default=None,
                    metavar="B,H,Hkv,Nk,d", help="decode workload (default 8,32,32,32768,128)")
    ap.add_argument("--link", action="store_true",
                    help="measure the host link for the end-to-end step's bytes instead")
    ap.add_argument("--deterministic", action="store_true",
                    help="time the deterministic backward (fa_bwd_deterministic) in the step")
    ap.add_argument("--shape", type=lambda x: tuple(int(v) for v in x.split(",")), default=None,
                    metavar="B,H,N,d",
                    help="run another shape (profiling captures on a smaller case); the metric "
                         "is defined on the default B=2,H=32,N=8192,d=128")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        world, rank, _ = dist_setup("gloo")
        run_reference(args, world, rank)
    else:
        world, rank, local = dist_setup("nccl")
        if args.link:
            run_link(args, world, rank, local)
        elif args.decode:
            run_decode(args, world, rank, local)
        elif args.fp8:
            run_fp8(args, world, rank, local)
        else:
            run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
