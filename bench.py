#!/usr/bin/env python3
"""Benchmark of the persistent FP16 GEMM (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gemm_f16|reference]
                    [--workload NAME] [--order grouped|row-major] [--cross-tile on|off]

A step is one gemm_f16 call (one persistent kernel launch) over the whole
workload; the default workload is M = N = 16384, K = 4096, A and B row-major
fp16 N(0,1), fp32 accumulate and output, grouped order with GROUP_SIZE_M = 8,
cross-tile pipelining on. ``value`` is the device-timed throughput (CUDA
events on the launching stream, inputs resident in HBM); ``e2e`` is the same
metric through ``HostPipeline`` with pinned host operands, host<->device
copies inside the timed region. Under torchrun every rank runs its own copy
of the workload on its own GPU (independent problems, weak scaling).

``--impl reference`` times the CPU oracle (the reference arm of this build) on
a bounded sample of the same workload.
"""
import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# P of the target: GB300 dense FP16 tensor peak per GPU, from the GB300 NVL72
# specification (360 PFLOP/s sparse FP16 for 72 GPUs, halved for dense).
SPEC_FP16_TFLOPS = 2500.0
TARGET_FRACTION = 0.70              # the headline goal: >= 70 % of P
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0


# The headline metric, as stated for this workload; both arms report it.
METRIC = "FP16 GEMM TFLOPS (2MNK/s) and % of GB300 dense FP16 peak"


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=500)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["gemm_f16", "reference"], default="gemm_f16")
    p.add_argument("--workload", default=None)
    p.add_argument("--order", choices=["grouped", "row-major"], default="grouped")
    p.add_argument("--group-size", type=int, default=8)
    p.add_argument("--cross-tile", choices=["on", "off"], default="on")
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--e2e-repeats", type=int, default=2,
                   help="timed e2e windows of --e2e-steps each; the fastest is reported, all are listed "
                        "(the host link is shared with the rest of the machine)")
    p.add_argument("--burst-launches", type=int, default=10,
                   help="launches of the short burst loop after the timed region (0: skip)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="approximate CPU time of the oracle sample")
    p.add_argument("--no-clocks", action="store_true")
    p.add_argument("--single-cta", action="store_true",
                   help="one-CTA 128x256 tiles instead of CTA-pair 256x256 tiles")
    p.add_argument("--sweep-reps", type=int, default=3,
                   help="repetitions of each study point (interleaved); the median is reported")
    p.add_argument("--sweep-rest", type=float, default=1.0,
                   help="seconds of rest before each timed study point")
    p.add_argument("--sweep", choices=["order", "ksweep", "kernel", "persistence", "cublas", "splitk", "packed",
                                       "outdtype", "ragged", "schedule", "tail"],
                   default=None,
                   help="print one JSON line per point of a study instead of the bench line")
    return p.parse_args(argv)


# ---------------------------------------------------------------- helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return {"bf16_tflops": FALLBACK_BF16_TFLOPS, "hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for rel in ("dense_gemm_gb300/csrc/gemm_kernel.cuh", "dense_gemm_gb300/csrc/gemm_pair.cuh",
                "dense_gemm_gb300/csrc/ptx.cuh", "dense_gemm_gb300/csrc/gemm_f16.cu"):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def recorded_traffic(workload_name, order, cross):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source for this workload and schedule; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    key = f"{workload_name}|{order}|cross={'on' if cross else 'off'}"
    e = d.get(key)
    if not e or e.get("kernel_source_sha256") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples with host timestamps."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id=None, period_ms=100):
        self.samples = []
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", str(period_ms)]
        if gpu_id:
            cmd += ["-i", str(gpu_id)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        inside = [s for (t, s) in self.samples if t0 <= t <= t1]
        used = inside
        if not used:  # timed region shorter than the sampling period: nearest samples
            near = sorted(self.samples, key=lambda ts: min(abs(ts[0] - t0), abs(ts[0] - t1)))
            used = [s for _, s in near[:2]]
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [num(s[1]) for s in used if num(s[1]) is not None]
        smax = [num(s[2]) for s in used if num(s[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in used for i in range(4) if s[5 + i].lower() == "active"})
        power = [num(s[3]) for s in used if num(s[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons,
                "power_w_max": max(power) if power else None,
                "samples": len(inside), "samples_near": len(used) - len(inside)}


def power_capped(clocks):
    """Did the clock samples of the timed loop show it running at the power
    limit (sw_power_cap active, or a median SM clock below 90 % of its max)?"""
    if not clocks:
        return False, "no clock samples"
    if "sw_power_cap" in clocks.get("reasons", []):
        return True, "the clock samples of the timed loop show sw_power_cap"
    mhz, top = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    if mhz and top and mhz < 0.9 * top:
        return True, f"the median SM clock of the timed loop ({mhz:g} MHz) is below 90 % of its max ({top:g})"
    return False, "the clock samples of the timed loop show neither sw_power_cap nor a lowered SM clock"


def roofline_peak(peaks, source, clocks):
    """(peak TFLOP/s, note): the measured cuBLAS bf16 peak for the regime the
    timed loop ran in: the sustained one when it ran at the power limit, else
    the burst one (fp16 and bf16 have the same nominal dense rate)."""
    burst = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
    sustained = float(peaks.get("bf16_tflops_sustained", 0.0)) or None
    capped, why = power_capped(clocks)
    regime = "sustained" if capped and sustained else "burst"
    peak = sustained if regime == "sustained" else burst
    return peak, (f"{source} cuBLAS bf16 {regime} peak (MEASURED_PEAKS.json) x nominal fp16/bf16 "
                  f"ratio 1.0; {regime} because {why}")


def target_line(value_per_gpu, bound_tflops):
    """The headline goal, stated on one P: the GB300 dense FP16 tensor peak."""
    return {"P_tflops": SPEC_FP16_TFLOPS,
            "P_source": "GB300 NVL72 specification: 360 PFLOP/s sparse FP16 / 72 GPUs / 2 (dense)",
            "frac_of_P": value_per_gpu / SPEC_FP16_TFLOPS, "goal_frac": TARGET_FRACTION,
            "met": value_per_gpu >= TARGET_FRACTION * SPEC_FP16_TFLOPS,
            "frac_of_min_P_BWxI": value_per_gpu / bound_tflops}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` across the ranks of the default process group
    (timings: the job takes as long as its slowest rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, flops_per_rank_step: float, steps: int, max_ms: float) -> float:
    """Whole-job TFLOP/s: every rank's work divided by the slowest rank's time."""
    return world * flops_per_rank_step * steps / (max_ms * 1e-3) / 1e12


def l2_note(w):
    total = 2 * (w.M * w.K + w.K * w.N) + 4 * w.M * w.N
    if total > 126 * 2 ** 20:
        return f"no flush: A+B+C = {total / 2 ** 30:.2f} GiB per step, larger than the 126 MiB L2"
    return f"L2-resident: A+B+C = {total / 2 ** 20:.1f} MiB per step (smaller than L2, no flush)"


def workload_config(w, args, extra=None):
    cfg = {"workload": w.describe(), "name": w.name, "M": w.M, "N": w.N, "K": w.K,
           "order": args.order, "group_size_m": args.group_size if args.order == "grouped" else None,
           "cross_tile": args.cross_tile == "on", "a_layout": w.a_layout, "b_layout": w.b_layout,
           "values": w.dist, "seed": w.seed,
           "l2": l2_note(w)}
    if extra:
        cfg.update(extra)
    return cfg


# ---------------------------------------------------------------- CPU oracle legs

def oracle_rows_timing(A, B, rows, threads):
    import numpy as np
    import oracle
    r = np.asarray(rows, dtype=np.int64)
    t0 = time.perf_counter()
    oracle.gemm_rows(A, B, rows=r, threads=threads)
    return time.perf_counter() - t0


def host_cpu():
    """CPU model and architecture of this host (for the CPU-baseline line)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    return {"model": model or platform.processor() or "unknown", "machine": platform.machine()}


def host_link_rates(h2d_bytes, d2h_bytes, dev, reps=3):
    """GB/s of one pinned-host <-> device copy of each size (best of `reps`)."""
    import torch
    host_in = torch.empty(h2d_bytes, dtype=torch.uint8, pin_memory=True)
    host_out = torch.empty(d2h_bytes, dtype=torch.uint8, pin_memory=True)
    dev_in = torch.empty(h2d_bytes, dtype=torch.uint8, device=dev)
    dev_out = torch.zeros(d2h_bytes, dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream(dev)

    def best(fn, nbytes):
        t = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            with torch.cuda.stream(s):
                fn()
            e1.record(s)
            s.synchronize()
            t.append(e0.elapsed_time(e1))
        return nbytes / (min(t) * 1e-3) / 1e9

    rates = {"h2d": best(lambda: dev_in.copy_(host_in, non_blocking=True), h2d_bytes),
             "d2h": best(lambda: host_out.copy_(dev_out, non_blocking=True), d2h_bytes)}
    del host_in, host_out, dev_in, dev_out
    return rates


def cpu_baseline(A, B, seconds):
    """Time the oracle, as it stands, on a bounded sample of whole C rows."""
    import numpy as np
    import oracle
    threads = os.cpu_count() or 1
    M, K = A.shape
    N = B.shape[1]
    rng = np.random.default_rng(0)
    probe = max(threads, 4)
    t_probe = oracle_rows_timing(A, B, rng.integers(0, M, probe), threads)
    rows = int(max(probe, min(M, probe * seconds / max(t_probe, 1e-6))))
    sample = rng.integers(0, M, rows)
    t = oracle_rows_timing(A, B, sample, threads)
    flops = 2.0 * rows * N * K
    return {"value": flops / t / 1e12, "unit": "TFLOP/s", "cores": int(oracle.max_threads()),
            "kind": "oracle", "host": host_cpu(),
            "sample": f"{rows} random rows of C (full N={N}, K={K}) = {rows / M:.4%} of the "
                      f"workload's FLOPs, {t:.1f} s on {threads} host threads"}


def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import numpy as np
    import oracle
    A, B = w.operands()
    threads = os.cpu_count() or 1
    M, K = A.shape
    N = B.shape[1]
    rng = np.random.default_rng(1)
    probe = max(threads, 4)
    t_probe = oracle_rows_timing(A, B, rng.integers(0, M, probe), threads)
    per_step_s = min(20.0, 150.0 / max(1, args.steps + args.warmup))
    rows = int(max(1, min(M, probe * per_step_s / max(t_probe, 1e-6))))
    for _ in range(args.warmup):
        oracle_rows_timing(A, B, rng.integers(0, M, rows), threads)
    times = [oracle_rows_timing(A, B, rng.integers(0, M, rows), threads) for _ in range(args.steps)]
    total = sum(times)
    flops_step = 2.0 * rows * N * K
    value = flops_step * args.steps / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value,
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, args, {"rows_per_step": rows}),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "kind": "oracle",
                         "cores": int(oracle.max_threads()), "host": host_cpu(),
                         "sample": f"each step: {rows} random whole rows of C "
                                   f"({rows / M:.4%} of the workload)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU leg

def run_gpu(args, w):
    import torch
    import torch.distributed as dist

    from dense_gemm_gb300 import HostPipeline, gemm, kernel_info, sync_status

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    grouped = args.order == "grouped"
    cross = args.cross_tile == "on"
    A_host, B_host = w.operands()
    A = A_host.to(dev)
    B = B_host.to(dev)
    C = torch.empty((w.M, w.N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        gemm(A, B, C, group_size_m=args.group_size, grouped=grouped, cross_tile=cross,
             single_cta=args.single_cta, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    if sync_status(stream) != 0:
        raise RuntimeError("device status after warm-up is not GEMM_OK")

    # one launch right after a 512 MiB write has flushed L2, next to the warm loop below
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    flush.fill_(1)
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    step()
    c1.record(stream)
    torch.cuda.synchronize(dev)
    cold_l2_ms = c0.elapsed_time(c1)
    del flush

    sampler = None
    if not args.no_clocks:
        props = torch.cuda.get_device_properties(dev)
        gpu_id = getattr(props, "uuid", None)
        gpu_id = f"GPU-{gpu_id}" if gpu_id is not None and not str(gpu_id).startswith("GPU-") else gpu_id
        sampler = ClockSampler(gpu_id, period_ms=20)
        time.sleep(0.6)   # let nvidia-smi start
        for _ in range(max(args.warmup, 3)):
            step()
        torch.cuda.synchronize(dev)

    K_steps = args.steps
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(K_steps + 1)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    ev[0].record(stream)
    for i in range(K_steps):
        step()
        ev[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    if world > 1:
        dist.barrier()
    status = sync_status(stream)
    per_launch_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(K_steps)]
    total_ms = max_over_ranks(ev[0].elapsed_time(ev[K_steps]), dev)
    clocks = sampler.summary(t_wall0, t_wall1) if sampler else None
    if sampler:
        sampler.stop()

    flops = 2.0 * w.M * w.N * w.K
    value = job_throughput(world, flops, K_steps, total_ms)
    avg_launch_ms = statistics.mean(per_launch_ms)
    med_launch_ms = statistics.median(per_launch_ms)
    achieved = flops / (avg_launch_ms * 1e-3) / 1e12

    # ---- burst: after a 2 s rest, a short loop below the power limit (for the
    # burst peak; the timed loop above runs at the limit)
    burst_ms = None
    if args.burst_launches > 0:
        time.sleep(2.0)
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        for _ in range(args.burst_launches):
            step()
        b1.record(stream)
        torch.cuda.synchronize(dev)
        burst_ms = b0.elapsed_time(b1) / args.burst_launches

    # ---- end to end: host operands, copies in the timed region
    e2e = None
    if not args.no_e2e and args.e2e_steps > 0:
        A_pin = A_host.pin_memory()
        B_pin = B_host.pin_memory()
        C_pin = torch.empty((w.M, w.N), dtype=torch.float32, pin_memory=True)
        del C  # the pipeline holds its own device buffers
        torch.cuda.empty_cache()
        in_bytes = A_host.untyped_storage().nbytes() + B_host.untyped_storage().nbytes()
        out_bytes = 4 * w.M * w.N
        link = host_link_rates(in_bytes, out_bytes, dev)
        pipe = HostPipeline(A, B, depth=2, group_size_m=args.group_size, grouped=grouped,
                            cross_tile=cross, single_cta=args.single_cta, device=dev)
        del A, B
        for _ in range(2):  # warm-up: both buffer sets
            pipe.submit(A_pin, B_pin, C_pin)
        pipe.synchronize()
        windows = []
        for _ in range(max(1, args.e2e_repeats)):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            if world > 1:
                dist.barrier()
            e0.record(pipe.s_in)
            for _ in range(args.e2e_steps):
                pipe.submit(A_pin, B_pin, C_pin)
            e1.record(pipe.s_out)
            pipe.synchronize()
            windows.append(max_over_ranks(e0.elapsed_time(e1), dev))
        e2e_ms = min(windows)
        e2e = {"value": job_throughput(world, flops, args.e2e_steps, e2e_ms), "unit": "TFLOP/s",
               "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": out_bytes,
               "link_gbs": link,
               # uploads and downloads of consecutive steps overlap: the slower direction bounds a step
               "link_bound_ms_per_step": max(in_bytes / link["h2d"], out_bytes / link["d2h"]) / 1e6,
               "steps": args.e2e_steps, "ms_per_step": e2e_ms / args.e2e_steps,
               "windows_ms_per_step": [x / args.e2e_steps for x in windows],
               "api": "dense_gemm_gb300.HostPipeline (pinned host A, B -> device, gemm_f16, "
                      "C -> pinned host; upload+GEMM of step i+1 overlap the download of step i)"}
        del pipe, A_pin, B_pin, C_pin

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    peaks, peak_src = load_peaks()
    peak, peak_note = roofline_peak(peaks, peak_src, clocks)
    burst_peak = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    compulsory = 2 * (w.M * w.K + w.K * w.N) + 4 * w.M * w.N
    intensity = flops / compulsory
    bound_tflops = min(SPEC_FP16_TFLOPS, hbm * 1e9 * intensity / 1e12)
    traffic = recorded_traffic(w.name, args.order, cross)
    info = kernel_info(0 if args.single_cta else 4)

    line = {
        "metric": METRIC,
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K_steps,
        "warmup": args.warmup, "ms_per_step": total_ms / K_steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": workload_config(w, args, {"parallelism": f"independent replicas x{world}",
                                            "accumulate": "f32", "output": "f32",
                                            "tiles": "one CTA, 128x256" if args.single_cta
                                            else "CTA pair (cta_group::2), 256x256"}),
        "target": target_line(value / world, bound_tflops),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic, "peak_source": peak_note,
                     "burst": ({"achieved": flops / (burst_ms * 1e-3) / 1e12, "peak": burst_peak,
                                "frac": flops / (burst_ms * 1e-3) / 1e12 / burst_peak,
                                "launches": args.burst_launches, "avg_launch_ms": burst_ms,
                                "note": "short loop after a 2 s rest, against the burst peak"}
                               if burst_ms else None),
                     "kernel": ("g16::gemm_f16_persistent<true,true>" if args.single_cta
                                else "g16::gemm_f16_pair<true,true,false>"),
                     "algorithmic_flops_per_launch": flops,
                     "avg_launch_ms": avg_launch_ms, "median_launch_ms": med_launch_ms,
                     "workload_roofline_tflops_min_P_BWxI": bound_tflops,
                     "compulsory_bytes": compulsory},
        "e2e": e2e,
        "gpu_launches": K_steps,
        "cold_l2_launch_ms": cold_l2_ms,
        "clocks": clocks,
        "kernel_resources": info,
        "device_status": status,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(A_host, B_host, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0 if status == 0 else 1


# ---------------------------------------------------------------- studies

def run_sweep(args):
    """Device-timed points of one study, one JSON line each:
    order  - grouped vs row-major tile order (8192^2 and 16384^2, K = 4096);
    ksweep - cross-tile on vs off, 16384^2, K in {128 ... 4096};
    kernel - CTA-pair vs one-CTA tiles on the headline workload;
    persistence - the pages' four variants (tiled / persistent x row-major /
                  grouped) at 8192^2 and 16384^2, K = 4096;
    cublas - context line: torch.matmul (cuBLAS, fp16 output) on 8192^2 and
             16384^2, K = 4096, next to gemm_f16 (fp32 C) and gemm_f16_out (fp16 C)
             on the same operands;
    splitk - gemm_f16 vs gemm_f16_splitk (automatic slices) on 512^3 and
             1024^2 x 32768 (fewer tiles than CTA pairs);
    outdtype - fp32 vs fp16 vs bf16 C (gemm_f16_out) on the headline workload
               and at K = 512, where the C store dominates the traffic;
    ragged - the two ragged workloads (4000 x 5000 x 3000 through TMA, 8191^2 x 257
             with 514-byte rows through the predicated-load path) and 512^3;
    schedule - the static pid + i*P tile stream vs GEMM_SCHED_DYNAMIC (cluster
               launch control) on 8192^2 x 4096, 16384^2 x 1024, 4000 x 5000 x 3000;
    tail - GEMM_SCHED_TAIL_SPLIT off/on (fp32 C, and fp16 C) with cuBLAS (fp16 C)
           beside, on 8192^2 x 4096, 4000 x 5000 x 3000, 512^3 and the headline;
    packed - gemm_f16 vs gemm_f16_packed (operands copied onto 128-byte lines
             first; with and without the split tail) on the ragged workloads and
             8192^2 x 4100 (8200-byte rows)."""
    import torch
    from dense_gemm_gb300 import (gemm, gemm_packed, gemm_splitk, packed_workspace_size, splitk_workspace_size,
                                  sync_status)
    from dense_gemm_gb300.inputs import HEADLINE, WORKLOADS

    dev = torch.device("cuda", 0)
    if args.sweep == "order":
        names = ["square_8192x8192x4096", HEADLINE]
        points = [dict(grouped=g, cross_tile=True, single_cta=False) for g in (True, False)]
    elif args.sweep == "ksweep":
        names = [n for n in WORKLOADS if n.startswith("ksweep_")]
        points = [dict(grouped=True, cross_tile=c, single_cta=False) for c in (True, False)]
    elif args.sweep == "ragged":
        names = ["ragged_4000x5000x3000", "ragged_8191x8191x257", "square_512"]
        points = [dict(grouped=True, cross_tile=True, single_cta=False)]
    elif args.sweep == "schedule":
        names = ["square_8192x8192x4096", "ksweep_16384x16384x1024", "ragged_4000x5000x3000"]
        points = [dict(grouped=True, cross_tile=True, single_cta=False, dynamic=d) for d in (False, True)]
    elif args.sweep == "tail":
        names = ["square_8192x8192x4096", "ragged_4000x5000x3000", "square_512", HEADLINE]
        points = [dict(grouped=True, cross_tile=True, single_cta=False, tail_split=t) for t in (False, True)]
        points += [("out", torch.float16), ("out16_tail", torch.float16), "torch.matmul"]
    elif args.sweep == "packed":
        names = ["ragged_4000x5000x3000", "ragged_8191x8191x257", "unaligned_8192x8192x4100"]
        points = [dict(grouped=True, cross_tile=True, single_cta=False), "packed", "packed_tail"]
    elif args.sweep == "outdtype":
        names = [HEADLINE, "ksweep_16384x16384x512"]
        points = [("out", torch.float32), ("out", torch.float16), ("out", torch.bfloat16)]
    elif args.sweep == "splitk":
        names = ["square_512", "longk_1024x1024x32768"]
        points = [dict(grouped=True, cross_tile=True, single_cta=False), "splitk"]
    elif args.sweep == "cublas":
        names = ["square_8192x8192x4096", HEADLINE]
        points = [dict(grouped=True, cross_tile=True, single_cta=False), ("out", torch.float16), "torch.matmul"]
    elif args.sweep == "persistence":
        names = ["square_8192x8192x4096", HEADLINE]
        points = [dict(grouped=g, cross_tile=True, single_cta=False, persistent=per)
                  for per in (False, True) for g in (False, True)]
    else:
        names = [HEADLINE]
        points = [dict(grouped=True, cross_tile=True, single_cta=s) for s in (False, True)]
    steps = max(args.steps, 1)
    for name in names:
        w = WORKLOADS[name]
        A_host, B_host = w.operands()
        A, B = A_host.to(dev), B_host.to(dev)
        C = torch.empty((w.M, w.N), dtype=torch.float32, device=dev)
        runs = []
        for pt in points:
            if isinstance(pt, tuple) and pt[0] in ("out", "out16_tail"):
                Cx = torch.empty((w.M, w.N), dtype=pt[1], device=dev)
                tail = pt[0] == "out16_tail"
                run = (lambda Cx=Cx, tail=tail:
                       gemm(A, B, Cx, group_size_m=args.group_size, tail_split=tail))
                desc = {"impl": "gemm_f16_out" if pt[1] != torch.float32 else "gemm_f16",
                        "c_dtype": str(pt[1]).replace("torch.", "")}
                if tail:
                    desc["tail_split"] = True
            elif pt == "torch.matmul":
                run = lambda: torch.matmul(A, B)  # noqa: E731  (cuBLAS, fp16 output)
                desc = {"impl": "torch.matmul (cuBLAS), fp16 output"}
            elif pt in ("packed", "packed_tail"):
                sam, sak = (max(x, 1) for x in A.stride())
                sbk, sbn = (max(x, 1) for x in B.stride())
                need = packed_workspace_size(w.M, w.N, w.K, sam, sak, sbk, sbn)
                ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
                tail = pt == "packed_tail"
                run = (lambda ws=ws, tail=tail:
                       gemm_packed(A, B, C, workspace=ws, group_size_m=args.group_size, tail_split=tail))
                desc = {"impl": "gemm_f16_packed", "tail_split": tail, "workspace_bytes": need}
            elif pt == "splitk":
                need, used = splitk_workspace_size(w.M, w.N, w.K, 0)
                ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
                run = (lambda ws=ws:
                       gemm_splitk(A, B, C, splits=0, workspace=ws, group_size_m=args.group_size))
                desc = {"impl": "gemm_f16_splitk", "splits": used, "workspace_bytes": need}
            else:
                run = lambda pt=pt: gemm(A, B, C, group_size_m=args.group_size, **pt)  # noqa: E731
                desc = {"impl": "gemm_f16", **pt, "group_size_m": args.group_size}
            runs.append((desc, run))
        # points interleaved, each repetition after a rest, so that every point
        # sees the same mix of power and clock states; the median is reported
        times = [[] for _ in runs]
        for _ in range(max(args.sweep_reps, 1)):
            for i, (desc, run) in enumerate(runs):
                time.sleep(args.sweep_rest)
                for _ in range(max(args.warmup, 3)):
                    run()
                torch.cuda.synchronize(dev)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(steps):
                    run()
                e1.record()
                torch.cuda.synchronize(dev)
                times[i].append(e0.elapsed_time(e1) / steps)
        flops = 2.0 * w.M * w.N * w.K
        for (desc, _), t in zip(runs, times):
            ms = statistics.median(t)
            print(json.dumps({"study": args.sweep, "workload": name, "M": w.M, "N": w.N, "K": w.K,
                              **desc, "steps": steps, "reps": len(t), "ms_per_launch": ms,
                              "ms_per_launch_reps": t, "tflops": flops / (ms * 1e-3) / 1e12,
                              "status": sync_status()}),
                  flush=True)
        del A, B, C
    return 0


def main(argv=None):
    args = parse_args(argv)
    from dense_gemm_gb300.inputs import HEADLINE, WORKLOADS
    if args.sweep:
        return run_sweep(args)
    w = WORKLOADS[args.workload or HEADLINE]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_gpu(args, w)


if __name__ == "__main__":
    sys.exit(main())
