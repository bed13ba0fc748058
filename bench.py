#!/usr/bin/env python3
"""Benchmark of the SRWM forward recurrence on GB300.

One step = one srwm_forward_balanced call over the whole workload (every row of the hot
path: input softmax when enabled, Eq. (1) read-out, phi of k and q, gates,
fused Eq. (2)/(3) update).  Default workload: "mid" (B=64, T=1024, H=8, d=64,
four learning rates), the d = 64 configuration the FP32-FMA target is stated
for, one GPU.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun (N > 1) every rank runs its own
copy of the workload on its own GPU (weak scaling, no data-path collective);
value = all ranks' head-tokens / max-over-ranks time.
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from self_referential_weight_gb300 import inputs  # noqa: E402

METRIC = "SRWM head-token updates/s (B*T*H/s) and % of FP32 FMA peak, 1 GB300"
UNIT = "head-token updates/s"
FMA_PER_CLK_PER_SM = 128          # FP32 FMA lanes per SM (4 SMSPs x 32)
L2_FLUSH_BYTES = 256 << 20        # > 129 MB L2
# Source files of each kernel; a committed ncu summary is used only while
# their hash matches the one recorded in it.
KERNEL_SOURCES = {
    "srwm_d64_kernel": ["srwm_d64.cuh", "srwm_ptx.cuh", "srwm_common.h", "srwm_d64.cu"],
    "srwm_d64r_kernel": ["srwm_d64r.cuh", "srwm_ptx.cuh", "srwm_common.h", "srwm_d64.cu"],
    "srwm_d32_kernel": ["srwm_d32.cuh", "srwm_ptx.cuh", "srwm_common.h", "srwm_d32.cu"],
    "srwm_d16_kernel": ["srwm_d16r.cuh", "srwm_ptx.cuh", "srwm_common.h", "srwm_d16.cu"],
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="mid", choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the device timing of the other workloads (long, rl, fewshot) on one GPU")
    ap.add_argument("--backward", action="store_true",
                    help="time srwm_backward (gradients of a loss on y) on the workload instead; prints its own line")
    ap.add_argument("--layer", action="store_true",
                    help="time one Recursive Self-Transformer layer (SRWM + LN + FF + residual, d_ff = 4D) "
                         "on the workload's shape instead; prints its own line")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(seconds, device=None):
    """Largest value over all ranks (the job's time is its slowest rank's);
    the value itself when not running distributed."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(seconds)
    t = torch.tensor([float(seconds)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_workload(wl, rank):
    """Weak scaling: every rank runs the same workload shape on its own seed."""
    return wl.with_shape(seed=wl.seed + 1000 * rank) if rank else wl


def fmas_per_head_token(wl):
    return 3 * wl.m * wl.d


def kernel_name(wl, n_sm):
    """The kernel the library launches for this workload (see srwm_d16.cu,
    srwm_d32.cu and srwm_d64.cu)."""
    if wl.d == 16:
        return "srwm_d16_kernel"
    if wl.d == 32:
        return "srwm_d32_kernel"
    return "srwm_d64r_kernel" if wl.B * wl.H > 2 * n_sm else "srwm_d64_kernel"


def profile_summary_path(kernel, workload):
    return os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")


def kernel_source_hash(kernel):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "self_referential_weight_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    this workload with the current kernel sources; else None."""
    try:
        text = open(profile_summary_path(kernel, workload)).read()
    except OSError:
        return None
    src = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    wl = re.search(r"workload:\s*(\w+)", text)
    tr = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    if not (src and wl and tr) or src.group(1) != kernel_source_hash(kernel) or wl.group(1) != workload:
        return None
    return int(tr.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle sampling around a timed region.

    Samples are read by a thread and time-stamped on arrival; entering waits
    for the first sample, so sampling is running when the timed region starts.
    summary(t0, t1) keeps the samples taken between t0 and t1 (wall clock),
    which the caller brackets around the timed region plus a short roll of
    the same work before and after it, so that a region of a few milliseconds
    still gets samples under load."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 50

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line))

    def __enter__(self):
        import threading

        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.INTERVAL_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t_end = time.time() + 5.0
        while not self.lines and time.time() < t_end and self.proc.poll() is None:
            time.sleep(0.01)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
            if self.thread is not None:
                self.thread.join(timeout=5)

    def summary(self, t0=None, t1=None):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in list(self.lines):
            if (t0 is not None and ts < t0) or (t1 is not None and ts > t1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


ROLL_S = 0.15   # seconds of untimed load on each side of a timed region while clocks are sampled


def one_call_ms(step, stream):
    """Device time of one call (for sizing the clock-sampling roll)."""
    import torch

    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    step()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b)


def roll(step, seconds, ms_per_call):
    """Runs `step` for about `seconds` of GPU time (untimed: it only keeps the
    GPU under the same load while clocks are sampled around a timed region)."""
    import torch

    for _ in range(max(1, int(seconds * 1e3 / max(ms_per_call, 1e-3)))):
        step()
    torch.cuda.synchronize()


def cpu_model():
    """The host CPU's vendor and model as lscpu or /proc/cpuinfo report them."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        info = {}
        for line in out.splitlines():
            k, _, v = line.partition(":")
            info.setdefault(k.strip(), v.strip())
        parts = [info.get("Vendor ID"), info.get("Model name")]
        if any(parts):
            return " ".join(p for p in parts if p)
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu model")):
                return line.partition(":")[2].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline(wl, x, W0, target_s=10.0):
    """The float64 oracle, as it stands, on this host's cores, on a bounded sample
    of the workload's (b, h) streams at full T.  Returns the JSON object."""
    import oracle

    cores = os.cpu_count() or 1
    # calibrate on a handful of streams, then size the sample to ~target_s
    n_cal = min(wl.B * wl.H, max(cores, 8))
    pairs = [(i // wl.H, i % wl.H) for i in range(wl.B * wl.H)]

    def run(n, threads=cores):
        sel = pairs[:n]
        xs = np.ascontiguousarray(np.stack([x[b, :, h] for b, h in sel], axis=0)[:, :, None, :])
        Ws = np.ascontiguousarray(np.stack([W0[h] for _, h in sel], axis=0)[:, None])
        t0 = time.perf_counter()
        oracle.forward(xs, Ws, wl.n_lr, wl.softmax_input, per_sequence=True, n_threads=threads)
        return time.perf_counter() - t0

    t_cal = run(n_cal)
    n = int(min(wl.B * wl.H, max(n_cal, n_cal * target_s / max(t_cal, 1e-6))))
    n = max(cores, (n // cores) * cores) if n >= cores else n
    n = min(n, wl.B * wl.H)
    dt = run(n)
    # the same oracle on one core, on a sample of ~3 s
    n1 = max(1, min(wl.B * wl.H, int(3.0 * n_cal / max(t_cal * cores, 1e-6))))
    dt1 = run(n1, threads=1)
    return {"value": n * wl.T / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} of {wl.B * wl.H} (b,h) streams x {wl.T} steps of the {wl.name} "
                      f"workload, float64 C oracle, one pthread per core over streams",
            "seconds": dt,
            "one_core": {"value": n1 * wl.T / dt1, "unit": UNIT, "cores": 1,
                         "sample": f"{n1} streams x {wl.T} steps, one thread", "seconds": dt1},
            "cpu_model": cpu_model()}


def reference_arm(args, wl):
    """--impl reference: the oracle timed on the host cores, each step a bounded
    sample of the workload."""
    import oracle

    x, W0 = inputs.make_inputs(wl)
    cores = os.cpu_count() or 1
    n = min(wl.B * wl.H, 2 * cores)
    sel = [(i // wl.H, i % wl.H) for i in range(n)]
    xs = np.ascontiguousarray(np.stack([x[b, :, h] for b, h in sel], axis=0)[:, :, None, :])
    Ws = np.ascontiguousarray(np.stack([W0[h] for _, h in sel], axis=0)[:, None])

    def step():
        oracle.forward(xs, Ws, wl.n_lr, wl.softmax_input, per_sequence=True, n_threads=cores)

    for _ in range(args.warmup):
        step()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
    tot = sum(times)
    value = n * wl.T * args.steps / tot
    sample = (f"{n} of {wl.B * wl.H} (b,h) streams x {wl.T} steps of the {wl.name} workload per "
              f"step, float64 C oracle, {cores} host threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(wl),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(wl):
    return {"workload": wl.name, "B": wl.B, "T": wl.T, "H": wl.H, "d": wl.d, "m": wl.m,
            "n_lr": wl.n_lr, "softmax_input": wl.softmax_input,
            "l2": "flushed between timed steps (256 MiB write)",
            "inputs": "seeded SplitMix64/Box-Muller synthetic, x ~ N(0,1), W0 ~ N(0,1/d)"}


def main():
    args = parse()
    rank, world, local = dist_env()
    wl = inputs.workload(args.workload)

    if args.layer:
        return bench_layer(args, wl)
    if args.backward:
        return bench_backward(args, wl)
    if args.impl == "reference":
        if rank == 0:
            reference_arm(args, wl)
        return

    import torch

    from self_referential_weight_gb300 import binding

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()

    # per-rank data: the same workload shape, a rank-specific seed (weak scaling)
    wl_r = rank_workload(wl, rank)
    x_np, W0_np = inputs.make_inputs(wl_r)
    x = torch.from_numpy(x_np).to(dev)
    W0 = torch.from_numpy(W0_np).to(dev)
    y = torch.empty_like(x)
    Wf = torch.empty((wl.B, wl.H, wl.m, wl.d), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    workspace = torch.empty(binding.srwm_forward_workspace_bytes(wl.B, wl.H), dtype=torch.uint8, device=dev)

    def step():
        binding.srwm_forward_balanced(x, W0, wl.n_lr, wl.softmax_input, y_out=y, W_final=Wf,
                                      workspace=workspace, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if binding.srwm_last_device_status(stream) != 0:
        raise RuntimeError("device status set during warm-up")

    est_ms = one_call_ms(step, stream)

    # ---------------- device-timed region: K steps, L2 flushed between steps;
    # clocks sampled over the region and a short roll of the same calls on
    # either side of it
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    with (clocks if not args.no_clocks else _Null()):
        t_roll0 = time.time()
        if not args.no_clocks:
            roll(step, ROLL_S, est_ms)
        barrier()
        torch.cuda.synchronize()
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
        barrier()
        t_wall = time.perf_counter() - t_wall
        if not args.no_clocks:
            roll(step, ROLL_S, est_ms)
        t_roll1 = time.time()
    per_step = [s.elapsed_time(e) for s, e in zip(starts, ends)]  # ms
    t_dev = sum(per_step) / 1e3
    if binding.srwm_last_device_status(stream) != 0:
        raise RuntimeError("device status set during the timed region")
    t_max = max_over_ranks(t_dev, dev)

    ht_per_step = wl.head_tokens
    value = world * ht_per_step * args.steps / t_max
    ms_per_step = 1e3 * t_max / args.steps

    # ---------------- end to end through the public API with host buffers:
    # srwm_forward_host copies x and W0 in and y and W_final out, overlapping
    # the copies with the recurrence chunk by chunk
    x_h = torch.from_numpy(x_np).pin_memory()
    W0_h = torch.from_numpy(W0_np).pin_memory()
    y_h = torch.empty(x_h.shape, dtype=torch.float32).pin_memory()
    Wf_h = torch.empty(tuple(Wf.shape), dtype=torch.float32).pin_memory()
    chunk = 0   # the library's plan: chunks doubling from 32 steps, an even middle, halving again at the end
    host_ws = torch.empty(binding.srwm_forward_host_workspace_bytes(wl.B, wl.T, wl.H, wl.d, wl.n_lr, chunk),
                          dtype=torch.uint8, device=dev)

    def e2e_step():
        binding.srwm_forward_host(x_h, W0_h, wl.n_lr, wl.softmax_input, y_out=y_h, W_final=Wf_h, chunk_steps=chunk,
                                  workspace=host_ws, stream=stream)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    t_e2e = max_over_ranks(e0.elapsed_time(e1) / 1e3, dev)
    e2e = {"value": world * ht_per_step * args.e2e_steps / t_e2e, "unit": UNIT,
           "h2d_bytes_per_step": x_h.numel() * 4 + W0_h.numel() * 4,
           "d2h_bytes_per_step": y_h.numel() * 4 + Wf_h.numel() * 4,
           "ms_per_step": 1e3 * t_e2e / args.e2e_steps, "api": "srwm_forward_host (chunks doubling from 32 steps, an even middle of at most max(256, T/8), halving at the end)"}
    # the host results agree with the device path's (chunk restarts change fp32
    # rounding only), within the parity bar for this length
    y_dev = y.cpu()
    e2e_dev = float((y_h - y_dev).abs().max()) / float(y_dev.abs().max())
    if e2e_dev > (1e-4 if wl.T <= 1024 else 1e-3):
        raise RuntimeError(f"e2e host results differ from the device results: {e2e_dev:.3g} relative")

    # ---------------- FMA probe (calibration of the FP32 roofline)
    props = torch.cuda.get_device_properties(dev)
    n_sm = props.multi_processor_count
    probe = fma_probe(binding, n_sm, stream)

    if rank != 0:
        return
    clk = clocks.summary(t_roll0, t_roll1) if not args.no_clocks else {"sm_mhz": None, "sm_max_mhz": None,
                                                        "reasons": ["unsampled"], "samples": 0}
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    f_max_mhz = float(peaks.get("sm_max_mhz") or clk.get("sm_max_mhz") or 2070.0)
    peak_tflops = n_sm * FMA_PER_CLK_PER_SM * 2 * f_max_mhz * 1e6 / 1e12
    flops_per_launch = 2.0 * fmas_per_head_token(wl) * ht_per_step
    kernel_s = statistics.fmean(per_step) / 1e3
    achieved = flops_per_launch / kernel_s / 1e12
    peak_load = (n_sm * FMA_PER_CLK_PER_SM * 2 * clk["sm_mhz"] * 1e6 / 1e12) if clk["sm_mhz"] else None
    line = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": workload_config(wl),
        "fma_peak_frac": achieved / peak_tflops,
        "roofline": {
            "bound": "alu",
            "achieved": achieved,
            "peak": peak_tflops,
            "unit": "TFLOP/s",
            "frac": achieved / peak_tflops,
            "traffic": profiled_traffic(kernel_name(wl, n_sm), wl.name),
            "kernel": kernel_name(wl, n_sm),
            "flops_per_launch": flops_per_launch,
            "peak_basis": f"{n_sm} SMs x {FMA_PER_CLK_PER_SM} FP32 FMA/clk x 2 flop x "
                          f"{f_max_mhz:.0f} MHz (max SM clock)",
            "frac_at_load_clock": (achieved / peak_load) if peak_load else None,
        },
        "fma_probe": probe,
        "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"],
                   "reasons": clk["reasons"], "samples": clk["samples"],
                   "window": f"nvidia-smi every {ClockSampler.INTERVAL_MS} ms over the timed region and "
                             f"{ROLL_S} s of the same calls on each side"},
        "e2e": e2e,
        "gpu_launches": args.steps,
        "wall_s_timed_region": t_wall,
        "ms_per_step_best": min(per_step),
        "ms_per_step_median": statistics.median(per_step),
    }
    if world == 1 and not args.no_extra:
        # the other workloads, each timed on the device the same way; the
        # headline value and config stay the workload above
        del x, W0, y, Wf
        torch.cuda.empty_cache()
        extra_steps = max(10, min(args.steps, 50))
        line["other_workloads"] = {
            name: time_other_workload(binding, name, extra_steps, args.warmup, dev, flush, not args.no_clocks, n_sm,
                                      peak_tflops)
            for name in ("mid", "long", "rl", "fewshot") if name != wl.name}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, x_np, W0_np)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def time_other_workload(binding, name, steps, warmup, dev, flush, sample_clocks, n_sm, peak_tflops):
    """Device time of srwm_forward_balanced on another workload (one GPU):
    K timed calls after W warm-ups, L2 flushed between calls, CUDA events on
    the launching stream, clocks sampled during the timed region."""
    import torch

    wl = inputs.workload(name)
    x_np, W0_np = inputs.make_inputs(wl)
    x, W0 = torch.from_numpy(x_np).to(dev), torch.from_numpy(W0_np).to(dev)
    y = torch.empty_like(x)
    Wf = torch.empty((wl.B, wl.H, wl.m, wl.d), dtype=torch.float32, device=dev)
    ws = torch.empty(binding.srwm_forward_workspace_bytes(wl.B, wl.H), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        binding.srwm_forward_balanced(x, W0, wl.n_lr, wl.softmax_input, y_out=y, W_final=Wf, workspace=ws,
                                      stream=stream)

    for _ in range(max(warmup, 3)):
        step()
    torch.cuda.synchronize()
    est_ms = one_call_ms(step, stream)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    clocks = ClockSampler(torch.cuda.current_device())
    with (clocks if sample_clocks else _Null()):
        t_roll0 = time.time()
        if sample_clocks:
            roll(step, ROLL_S, est_ms)
        for i in range(steps):
            flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
        if sample_clocks:
            roll(step, ROLL_S, est_ms)
        t_roll1 = time.time()
    if binding.srwm_last_device_status(stream) != 0:
        raise RuntimeError(f"device status set while timing {name}")
    per_step = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    ms = statistics.fmean(per_step)
    flops = 2.0 * fmas_per_head_token(wl) * wl.head_tokens
    achieved = flops / (ms / 1e3) / 1e12
    kernel = kernel_name(wl, n_sm)
    clk = clocks.summary(t_roll0, t_roll1) if sample_clocks else {"sm_mhz": None, "sm_max_mhz": None,
                                                                  "reasons": ["unsampled"],
                                                  "samples": 0}
    return {"config": workload_config(wl), "steps": steps, "ms_per_step": ms,
            "ms_per_step_best": min(per_step), "ms_per_step_median": statistics.median(per_step),
            "value": wl.head_tokens / (ms / 1e3), "unit": UNIT,
            "roofline": {"bound": "alu", "achieved": achieved, "peak": peak_tflops, "unit": "TFLOP/s",
                         "frac": achieved / peak_tflops, "traffic": profiled_traffic(kernel, wl.name),
                         "kernel": kernel, "flops_per_launch": flops},
            "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"],
                       "samples": clk["samples"]}}


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *exc):
        return False


def fma_probe(binding, n_sm, stream):
    """FP32 FMA throughput of the calibration kernel (scalar and two-wide)."""
    import torch

    threads, iters = 512, 4096
    blocks = n_sm * 4
    out = torch.empty(blocks * threads, dtype=torch.float32, device="cuda")
    res = {}
    for packed in (0, 1):
        binding.srwm_probe_fma(blocks, threads, iters, packed, out, stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        reps = 5
        for _ in range(reps):
            binding.srwm_probe_fma(blocks, threads, iters, packed, out, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        s = e0.elapsed_time(e1) / 1e3 / reps
        fmas = blocks * threads * iters * 8 * (2 if packed else 1)
        res["tflops_packed" if packed else "tflops_scalar"] = 2 * fmas / s / 1e12
    return res


def bench_backward(args, wl):
    """srwm_backward on the workload: dL/dx and dL/dW0 of L = <dy, y> (1 GPU,
    L2 flushed between timed calls).  One call runs the forward with its
    per-step records, then the steps backwards; its arithmetic is 3md (forward)
    + 7md (backward step) FMAs per head-token."""
    import torch
    from self_referential_weight_gb300 import binding

    dev = torch.device("cuda:0")
    x_np, W0_np = inputs.make_inputs(wl)
    dy_np, _ = inputs.make_cotangents(wl, False)
    x, W0, dy = (torch.from_numpy(a).to(dev) for a in (x_np, W0_np, dy_np))
    dx, dW0 = torch.empty_like(x), torch.empty_like(W0)
    ws = torch.empty(binding.srwm_backward_workspace_bytes(wl.B, wl.T, wl.H, wl.d, wl.n_lr), dtype=torch.uint8,
                     device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def call():
        binding.srwm_backward(x, W0, wl.n_lr, wl.softmax_input, dy, None, dx, dW0, ws)

    for _ in range(max(args.warmup, 3)):
        call()
    torch.cuda.synchronize()
    steps = max(3, min(args.steps, 20))
    ts = []
    for _ in range(steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        call()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    if binding.srwm_last_device_status() != 0:
        raise RuntimeError("device status set")
    t = statistics.median(ts)
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    peak = n_sm * FMA_PER_CLK_PER_SM * 2 * 2070e6 / 1e12
    flops = 2 * 10 * wl.m * wl.d * wl.head_tokens
    print(json.dumps({
        "metric": "SRWM backward (dL/dx, dL/dW0), head-token gradients/s (1 GB300)",
        "value": wl.head_tokens / (t / 1e3), "unit": "head-token gradients/s", "ms_per_step": t, "steps": steps,
        "config": workload_config(wl), "dtype": "f32", "data": "synthetic",
        "fp32_fma_frac": flops / (t / 1e3) / 1e12 / peak,
        "fma_basis": "3md forward + 7md backward FMAs per head-token; 2070 MHz peak",
        "workspace_bytes": ws.numel(),
    }), flush=True)


def bench_layer(args, wl):
    """One Recursive Self-Transformer layer on the workload's shape: tokens/s
    of srwm_layer_forward, its SRWM part alone, and the feed-forward GEMMs with
    emulated and plain FP32 (1 GPU, L2 flushed between timed calls)."""
    import torch
    from self_referential_weight_gb300 import binding

    dev = torch.device("cuda:0")
    D, d_ff = wl.H * wl.d, 4 * wl.H * wl.d
    p = {k: torch.from_numpy(v).to(dev) for k, v in inputs.make_layer_params(wl.H, wl.d, wl.n_lr, d_ff, wl.seed).items()}
    u = torch.from_numpy(inputs.make_layer_input(wl.B, wl.T, D, wl.seed)).to(dev)
    out = torch.empty_like(u)
    ws = torch.empty(binding.srwm_layer_workspace_bytes(wl.B, wl.T, wl.H, wl.d, wl.n_lr, d_ff), dtype=torch.uint8,
                     device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def layer():
        binding.srwm_layer_forward(u, wl.H, wl.n_lr, wl.softmax_input, p["ln1_gamma"], p["ln1_beta"], p["W0"],
                                   p["ln2_gamma"], p["ln2_beta"], p["W1"], p["b1"], p["W2"], p["b2"], out=out,
                                   workspace=ws)

    x4 = u.view(wl.B, wl.T, wl.H, wl.d)
    y = torch.empty_like(x4)
    Wf = torch.empty((wl.B, wl.H, wl.m, wl.d), device=dev)
    cnt = torch.empty(binding.srwm_forward_workspace_bytes(wl.B, wl.H), dtype=torch.uint8, device=dev)

    def srwm():
        binding.srwm_forward_balanced(x4, p["W0"], wl.n_lr, wl.softmax_input, y_out=y, W_final=Wf, workspace=cnt)

    def timed(fn, steps):
        for _ in range(max(args.warmup, 3)):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        if binding.srwm_last_device_status() != 0:
            raise RuntimeError("device status set")
        return statistics.median(ts)

    steps = max(3, min(args.steps, 20))
    t_layer = timed(layer, steps)
    t_srwm = timed(srwm, steps)
    t_cmp = {}
    for mode, name in ((2, "cublaslt_emulated_fp32"), (1, "cublaslt_plain_fp32")):
        binding.srwm_debug_set_layer_gemm(mode)
        try:
            t_cmp[name] = timed(layer, steps)
        finally:
            binding.srwm_debug_set_layer_gemm(0)
    tokens = wl.B * wl.T
    ff_flops = 2 * 2 * tokens * D * d_ff
    ff_ms = t_layer - t_srwm
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    sustained = peaks.get("bf16_tflops_sustained")
    # the tensor cores run three bf16 products per fp32 product (hi*hi, hi*lo, lo*hi)
    tc_tflops = 3 * ff_flops / (ff_ms / 1e3) / 1e12
    print(json.dumps({
        "metric": "Recursive Self-Transformer layer forward, tokens/s (1 GB300)",
        "value": tokens / (t_layer / 1e3), "unit": "tokens/s", "ms_per_step": t_layer, "steps": steps,
        "config": {"workload": wl.name, "B": wl.B, "T": wl.T, "H": wl.H, "d": wl.d, "D": D, "d_ff": d_ff,
                   "n_lr": wl.n_lr, "softmax_input": wl.softmax_input, "l2": "flushed between timed steps"},
        "dtype": "f32", "data": "synthetic",
        "parts_ms": {"srwm_forward_alone": t_srwm, "layer_minus_srwm": ff_ms},
        "ff_gemm_flops": ff_flops,
        "ff_plus_ln_tflops_fp32_equivalent": ff_flops / (ff_ms / 1e3) / 1e12,
        "ff_plus_ln_bf16_tensor_tflops": tc_tflops,
        "ff_plus_ln_frac_of_bf16_sustained": (tc_tflops / sustained) if sustained else None,
        "comparison_ms_per_step": t_cmp,
    }), flush=True)

if __name__ == "__main__":
    main()
