#!/usr/bin/env python
"""SGEMM benchmark: GFLOP/s (2MNK / device time) of C = alpha*A*B + beta*C.

Default workload: the 8192^3 fp32 SGEMM (A, B uniform[-1,1], C_old normal,
alpha = 0.75, beta = 0.25, seed 2) through libphobos_gemm's default plan
(split TF32 on the tcgen05 tensor cores).  One "step" is one full call: the
split of A and B into tf32 pairs (by the main kernel itself for this shape)
and the GEMM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--math M]
  python bench.py --impl reference ...   # the CPU oracle, timed on the host cores

Prints ONE JSON line on rank 0.  Under torchrun (N > 1) every rank runs an
independent replica of the workload on its own GPU (the path does not shard);
the timed region is bracketed by barriers and the max over ranks is taken.
"""
import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SGEMM GFLOP/s (2MNK/device time) at 8192^3 fp32; fraction of GB300 roofline"
NOMINAL_TF32_OVER_BF16 = 1.1 / 2.25   # dense tensor rates, nominal
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
SMS, FP32_LANES_PER_SM = 152, 128
# --split: the plan's a_split values
SPLITS = {"auto": 0, "prepass": 1, "smem": 2, "kernel": 3}


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["phobos", "reference"], default="phobos")
    ap.add_argument("--workload", default="sgemm_8192")
    ap.add_argument("--math", default="default",
                    choices=["default", "3xtf32", "tf32", "ffma", "fp16", "bf16"])
    ap.add_argument("--multicast", action="store_true",
                    help="device-resident steps use the plan's multicast clusters (two CTA "
                         "pairs sharing A); the e2e leg keeps the automatic plan.  One GPU "
                         "only: refused under a multi-rank launch")
    ap.add_argument("--split", default="auto", choices=sorted(SPLITS),
                    help="where split TF32 splits A and B (the plan's a_split): the planner's "
                         "choice, a pre-pass, A in shared memory (B by the pre-pass), or the "
                         "main kernel's splitter warps.  The e2e leg keeps the automatic plan")
    ap.add_argument("--clc", action="store_true",
                    help="device-resident steps deal tiles to CTA pairs through Cluster Launch "
                         "Control (plan clc = 1, split TF32 only) instead of the static "
                         "persistent walk; the e2e leg keeps the automatic plan")
    ap.add_argument("--e2e-steps", type=int, default=10,
                    help="timed calls of the host-buffer leg (after one untimed call); their "
                         "mean is the e2e rate")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target host time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--reference-budget", type=float, default=150.0,
                    help="seconds the whole --impl reference run may take")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return d, "measured"
    except (OSError, ValueError):
        return {"bf16_tflops": FALLBACK_BF16_TFLOPS, "hbm_gbs": FALLBACK_HBM_GBS,
                "sm_max_mhz": 2070.0}, "fallback"


def peak_for(path_name, peaks):
    """Roofline denominator of the main kernel, by path."""
    if path_name in ("fp16", "bf16"):
        # 16-bit inputs run at the dense bf16/fp16 rate: the measured bf16 peak itself
        return ("tensor", peaks["bf16_tflops"], "TFLOP/s", "bf16 burst (fp16 has the same dense rate)")
    if path_name in ("3xtf32", "tf32"):
        tf32 = peaks["bf16_tflops"] * NOMINAL_TF32_OVER_BF16
        return ("tensor", tf32 / 3.0 if path_name == "3xtf32" else tf32, "TFLOP/s",
                "bf16 burst x nominal tf32/bf16 (1.1/2.25)%s" % (" / 3" if path_name == "3xtf32" else ""))
    mhz = peaks.get("sm_max_mhz", 2070.0)
    return ("alu", SMS * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12, "TFLOP/s",
            "152 SMs x 128 fp32 lanes x 2 flop x max SM clock")


def kernel_traffic(kernel_file, workload, math_name, multicast=False):
    """DRAM bytes per launch of the main kernel from the committed ncu summary,
    or None when the kernel source changed since the counters were taken."""
    if math_name == "ffma":
        summary = os.path.join(ROOT, "profiles", "sgemm_ffma_%s.md" % workload)
    else:
        summary = os.path.join(ROOT, "profiles", "sgemm_tc_%s%s_%s.md"
                               % (math_name, "_multicast" if multicast else "", workload))
    try:
        text = open(summary).read()
    except OSError:
        return None
    m_sha = re.search(r"kernel_source_sha256:\s*([0-9a-f]{64})", text)
    m_tr = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    if not m_sha or not m_tr:
        return None
    if kernel_source_sha256(kernel_file) != m_sha.group(1):
        return None
    return int(m_tr.group(1))


def code_only(text):
    """C/C++ source with comments removed and every run of whitespace outside
    string and character literals collapsed to one space, so that editing a
    comment or re-indenting leaves it unchanged."""
    out, code = [], []
    i, n = 0, len(text)

    def flush():
        if code:
            out.append(" ".join("".join(code).split()))
            code.clear()
    while i < n:
        c = text[i]
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
            code.append(" ")
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            code.append(" ")
        elif c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            flush()
            out.append(text[i:j + 1])
            i = j + 1
        else:
            code.append(c)
            i += 1
    flush()
    return " ".join(x for x in out if x)


def kernel_source_sha256(kernel_file):
    """SHA-256 over the code (comments and layout stripped, see code_only) of
    the kernel's source and the two headers it is built from."""
    h = hashlib.sha256()
    for name in (kernel_file, "ptx.cuh", "internal.h"):
        with open(os.path.join(ROOT, "language_fp32_gemm_gb300", "csrc", name)) as f:
            h.update(code_only(f.read()).encode())
            h.update(b"\0")
    return h.hexdigest()


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, with wall timestamps."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id):
        self.samples = []
        self.proc = None
        self.gpu_id = gpu_id

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
               "-lms", "20"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.samples and time.time() - t0 < 5.0:
            time.sleep(0.05)

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t_begin, t_end):
        rows = [s for t, s in self.samples if t_begin <= t <= t_end and len(s) >= 8]
        inside = len(rows)
        if not rows:  # a region shorter than the sampling interval: the nearest samples
            mid = 0.5 * (t_begin + t_end)
            near = sorted((abs(t - mid), i) for i, (t, s) in enumerate(self.samples)
                          if len(s) >= 8)[:2]
            rows = [self.samples[i][1] for _, i in sorted(near, key=lambda x: x[1])]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        pw = [num(r[2]) for r in rows if num(r[2]) is not None]
        reasons = sorted({name for r in rows for name, v in zip(self.REASONS, r[4:8])
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": reasons, "samples": len(rows), "samples_inside": inside}


def oracle_rows_rate(w, A, B, C0, seconds):
    """Time the CPU oracle on a row sample of the workload sized to ~seconds.

    Returns (GFLOP/s, rows used, threads, seconds taken)."""
    import oracle
    threads = oracle.default_threads()
    rows = max(1, min(w.M, threads))
    while True:
        t0 = time.perf_counter()
        oracle.sgemm(A[:rows], B, None if w.beta == 0 else C0[:rows], w.alpha, w.beta,
                     nthreads=threads)
        dt = time.perf_counter() - t0
        if dt >= seconds * 0.5 or rows >= w.M:
            return 2.0 * rows * w.N * w.K / dt / 1e9, rows, threads, dt
        grow = max(2.0, min(16.0, seconds * 0.8 / max(dt, 1e-3)))
        rows = min(w.M, int(math.ceil(rows * grow)))


def aggregate_rate(local_ms, flops_per_rank, steps, world, device=None):
    """Whole-job rate over `world` independent replicas: every rank processed
    `steps` problems of `flops_per_rank`; the job's time is the slowest rank's.
    Returns (max_ms, GFLOP/s).  Collective only when world > 1."""
    import torch
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    max_ms = float(t.item())
    return max_ms, world * flops_per_rank * steps / (max_ms / 1e3) / 1e9


# ------------------------------------------------------------- reference arm

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    import seeded_inputs as si
    w = si.workload(args.workload)
    A, B = w.A(), w.B()
    C0 = w.C_old() if w.beta != 0 else None
    threads = oracle.default_threads()
    per_step = max(0.5, args.reference_budget / max(1, args.steps + args.warmup))
    # calibrate rows per step on one probe
    rows = max(1, threads)
    t0 = time.perf_counter()
    oracle.sgemm(A[:rows], B, None if C0 is None else C0[:rows], w.alpha, w.beta, nthreads=threads)
    dt = time.perf_counter() - t0
    rows = int(max(1, min(w.M, rows * per_step / max(dt, 1e-3))))
    times = []
    for step in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.sgemm(A[:rows], B, None if C0 is None else C0[:rows], w.alpha, w.beta,
                     nthreads=threads)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            times.append(dt)
    flops = 2.0 * rows * w.N * w.K
    mean = sum(times) / len(times)
    value = flops / mean / 1e9
    sample = "%d of %d output rows per step (%dx%dx%d), fp64 oracle, %d threads" % (
        rows, w.M, w.M, w.N, w.K, threads)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": mean * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "M": w.M, "N": w.N, "K": w.K, "alpha": w.alpha,
                   "beta": w.beta, "seed": w.seed, "sample_rows": rows},
        "cpu_baseline": {"value": value, "unit": "GFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm

def run_phobos(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import language_fp32_gemm_gb300 as phobos
    import seeded_inputs as si

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    phobos.library()  # fails loudly if the CUDA library is not built

    w = si.workload(args.workload)
    M, N, K = w.M, w.N, w.K
    A_h, B_h, C_h = w.A(), w.B(), w.C_old()
    pin = lambda x: torch.from_numpy(x).pin_memory()
    A_p, B_p, C_p = pin(A_h), pin(B_h), pin(C_h)
    dA, dB = A_p.to(dev), B_p.to(dev)
    dC0 = C_p.to(dev)
    dC = dC0.clone()
    plan = phobos.phobos_gemm_plan(M, N, K, K, N, N, args.math)
    if args.multicast:
        plan.multicast, plan.cluster_n = 1, 2
    plan.a_split = SPLITS[args.split]
    plan.clc = 1 if args.clc else 0
    own_plan = args.multicast or args.split != "auto" or args.clc
    path_name = {phobos.PHOBOS_PATH_FFMA: "ffma", phobos.PHOBOS_PATH_TF32: "tf32",
                 phobos.PHOBOS_PATH_3XTF32: "3xtf32", phobos.PHOBOS_PATH_FP16: "fp16",
                 phobos.PHOBOS_PATH_BF16: "bf16"}[plan.path]
    stream = torch.cuda.current_stream(dev)

    def step():
        phobos.sgemm(dA, dB, dC, w.alpha, w.beta, math=args.math, stream=stream,
                     plan=plan if own_plan else None)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = phobos.phobos_check_device(stream.cuda_stream)
    if st != phobos.PHOBOS_OK:
        raise SystemExit("device status after warm-up: " + phobos.status_string(st))

    # per-step events around the main kernel (recorded by the library) and the step
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for a, b in kev:
        a.record(stream)
        b.record(stream)
    t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None
    clocks = ClockSampler(uuid) if rank == 0 else None
    if clocks:
        clocks.start()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = phobos.phobos_kernel_launches()
    phobos.phobos_kernel_clock_mhz()  # clear the kernels' cycle sum
    wall0 = time.time()
    t_start.record(stream)
    for i in range(args.steps):
        phobos.phobos_set_timing_events(kev[i][0].cuda_event, kev[i][1].cuda_event)
        step()
    phobos.phobos_set_timing_events(None, None)
    t_stop.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launches = phobos.phobos_kernel_launches() - launches0
    kernel_mhz = phobos.phobos_kernel_clock_mhz() or None  # tensor-core kernels only
    if clocks:
        clocks.stop()
    st = phobos.phobos_check_device(stream.cuda_stream)
    if st != phobos.PHOBOS_OK:
        raise SystemExit("device status after timed region: " + phobos.status_string(st))

    elapsed_ms = t_start.elapsed_time(t_stop)
    kernel_ms = [a.elapsed_time(b) for a, b in kev]
    flops = 2.0 * M * N * K
    max_ms, value = aggregate_rate(elapsed_ms, flops, args.steps, world, dev)

    # ------------------------------------------------ end to end, host buffers
    C_out = torch.empty_like(C_p).pin_memory()
    e2e_ms = []
    # --e2e-steps 0 skips this leg (profiling commands that capture only the
    # device-resident steps); the line's e2e is then null.
    for i in range(args.e2e_steps + 1 if args.e2e_steps > 0 else 0):
        C_out.copy_(C_p)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        st = phobos.phobos_sgemm_host(M, N, K, w.alpha, A_p.data_ptr(), K, B_p.data_ptr(), N,
                                      w.beta, C_out.data_ptr(), N, stream.cuda_stream,
                                      args.math)
        e1.record(stream)
        torch.cuda.synchronize()
        if st != phobos.PHOBOS_OK:
            raise SystemExit("phobos_sgemm_host: " + phobos.status_string(st))
        if i > 0:
            e2e_ms.append(e0.elapsed_time(e1))
    h2d = 4 * (M * K + K * N + (M * N if w.beta != 0 else 0))
    d2h = 4 * M * N
    e2e_value = None
    if e2e_ms:
        _, e2e_value = aggregate_rate(sum(e2e_ms) / len(e2e_ms), flops, 1, world, dev)

    if world > 1:
        dist.barrier()
    if rank != 0:
        dist.destroy_process_group()
        return 0

    # ------------------------------------------------------------- roofline
    peaks, peak_src = load_peaks()
    bound, peak, unit, peak_note = peak_for(path_name, peaks)
    kernel_file = "sgemm_ffma.cu" if path_name == "ffma" else "sgemm_tc.cu"
    avg_kernel_ms = sum(kernel_ms) / len(kernel_ms)
    achieved = flops / (avg_kernel_ms / 1e3) / 1e12
    clk = clocks.summary(wall0, wall1) if clocks else None
    # Per-clock view: nominal dense tensor rate per SM (tf32: 4096 flop/clk/SM,
    # i.e. 1.1 PFLOP/s at ~1.77 GHz; fp16/bf16: 8192) at the SM clock the
    # kernels counted themselves (cycles over global-timer time), else the one
    # nvidia-smi sampled.  Under the power cap the clock moves faster than
    # nvidia-smi samples it.
    per_clock = None
    per_clock_mhz = kernel_mhz or (clk.get("sm_mhz") if clk else None)
    if bound == "tensor" and per_clock_mhz:
        tf32_clk = SMS * 4096 * per_clock_mhz * 1e6 / 1e12
        per_clock = {"3xtf32": tf32_clk / 3.0, "tf32": tf32_clk}.get(path_name, 2 * tf32_clk)
    roofline = {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                # the committed counters are of the automatic split
                "frac": achieved / peak,
                "traffic": kernel_traffic(kernel_file, args.workload, path_name, args.multicast)
                           if args.split == "auto" and not args.clc else None,
                "peak_source": "%s (%s)" % (peak_src, peak_note),
                "kernel": "sgemm_tc_kernel" if path_name != "ffma" else "sgemm_ffma_kernel",
                "kernel_ms": avg_kernel_ms,
                "algorithmic_flops_per_launch": flops,
                "peak_per_clock": per_clock,
                "kernel_sm_mhz": kernel_mhz,
                "per_clock_mhz_source": ("kernel cycle counter" if kernel_mhz else
                                         "nvidia-smi median") if per_clock else None,
                "frac_per_clock": achieved / per_clock if per_clock else None}

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        rate, rows, threads, dt = oracle_rows_rate(w, A_h, B_h, C_h, args.cpu_seconds)
        cpu = {"value": rate, "unit": "GFLOP/s", "cores": threads, "kind": "oracle",
               "sample": "%d of %d output rows of the %dx%dx%d workload (fp64 oracle), %.1f s"
                         % (rows, M, M, N, K, dt)}

    line = {
        "metric": METRIC, "value": value, "unit": "GFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": max_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        # arithmetic of the path: tf32 products with fp32 accumulation (x3 for
        # the split), fp16 / bf16 products with fp32 accumulation, or fp32
        # fused multiply-add
        "dtype": {"3xtf32": "3xtf32", "tf32": "tf32", "ffma": "f32", "fp16": "f16",
                  "bf16": "bf16"}[path_name],
        "data": "synthetic",
        "config": {"workload": args.workload, "M": M, "N": N, "K": K, "alpha": w.alpha,
                   "beta": w.beta, "seed": w.seed, "math": path_name,
                   "plan": plan.as_dict(), "split": args.split, "clc": bool(args.clc),
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "inputs larger than L2 (%.0f MiB of A, B, C)"
                         % (4 * (M * K + K * N + M * N) / 2 ** 20),
                   "step": "one library call: split of A and B into tf32 pairs (inside the "
                           "main kernel, or a pre-pass, as the plan chooses) + the GEMM"},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "GFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": sum(e2e_ms) / len(e2e_ms),
                "steps": len(e2e_ms), "api": "phobos_sgemm_host (pinned host buffers)"}
               if e2e_ms else None,
        "gpu_launches": int(launches),
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    _, world, _ = dist_env()
    if args.multicast and (world > 1 or args.gpus > 1):
        # TMA multicast is a one-GPU option (its tensor maps cover this GPU's
        # own memory only): never part of a multi-GPU run.
        print("bench.py: --multicast runs on one GPU only (WORLD_SIZE=%d, --gpus %d)"
              % (world, args.gpus), file=sys.stderr, flush=True)
        return 2
    if args.impl == "reference":
        return run_reference(args)
    return run_phobos(args)


if __name__ == "__main__":
    sys.exit(main())
