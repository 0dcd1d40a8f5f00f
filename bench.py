#!/usr/bin/env python
"""W4A16 GEMM benchmark on GB300.

Default workload: the single large layer K=18432, N=73728, group 128, swept
over batch sizes M in {1, 2, 4, 8, 16, 32, 64, 128}.  One "step" runs the
GEMM once per M (the whole hot path over one batch of synthetic inputs per
M).  The packed weights (679 MB) exceed the 129 MB L2, so every GEMM streams
its weights from HBM without any flush.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload big|pr1|7b|70b|prefill|profile_m32|profile_m8|profile_m16]

Prints one JSON line (rank 0).  ``value`` is the whole-job throughput in TB/s
of algorithmic bytes (2MK + 0.5KN + 2(K/G)N + 2MN per GEMM) over the timed
region; ``sweep`` gives per-M microseconds, TB/s, TFLOP/s, the fraction of
the roofline max(bytes / HBM BW, FLOPs / dense FP16 peak), the kernel that
ran, and for context a cuBLAS FP16 GEMM (FP32 accumulation) on the
dequantised weights.  ``roofline`` describes the kernel with the largest share
of the step's device time (``roofline_by_kernel`` lists every kernel).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "W4A16 GEMM µs, achieved HBM TB/s & % of roofline vs M=1..128 (1×GB300)"
KERNEL_OF_PATH = {1: "gemm_mma_kernel", 2: "gemm_tc_kernel"}
L2_BYTES = 129 * 1024 * 1024
# roofline time below which a GEMM is also timed inside a CUDA graph (there the host's launch
# overhead, not the kernel, sets a single launch's time), and the minimum launches in that graph
GRAPH_BELOW_US = 20.0
GRAPH_LAUNCHES = 20
# columns of the first layer on which the oracle's repack is timed for the CPU baseline
REPACK_SAMPLE_COLS = 1024

# workload name -> (description, list of (K, N, groupsize, [M ...]), seed)
WORKLOADS = {
    "big": ("single large layer K=18432 N=73728 group 128, M sweep 1..128",
            [(18432, 73728, 128, [1, 2, 4, 8, 16, 32, 64, 128])], 2),
    "pr1": ("PR1: M=16 K=1024 N=1024 group 128", [(1024, 1024, 128, [16])], 0),
    "7b": ("7B-style decode layers, M in {1,16}, group 128",
           [(4096, 12288, 128, [1, 16]), (4096, 4096, 128, [1, 16]), (4096, 22016, 128, [1, 16]),
            (11008, 4096, 128, [1, 16])], 1),
    "70b": ("70B-style layers M=32, group 128 and per-column",
            [(8192, 10240, 128, [32]), (8192, 8192, 128, [32]), (8192, 57344, 128, [32]), (28672, 8192, 128, [32]),
             (8192, 10240, -1, [32]), (8192, 8192, -1, [32]), (8192, 57344, -1, [32]), (28672, 8192, -1, [32])], 3),
    "prefill": ("compute-bound prefill M in {256,512,1024}, K=8192 N=28672 group 128",
                [(8192, 28672, 128, [256, 512, 1024])], 4),
    # small cases of the big layer's kernels for full ncu captures (weights still larger than L2)
    "profile_m32": ("profiling case M=32 K=18432 N=16384 group 128", [(18432, 16384, 128, [32])], 2),
    "profile_m8": ("profiling case M=8 K=18432 N=16384 group 128", [(18432, 16384, 128, [8])], 2),
    "profile_m16": ("profiling case M=16 K=18432 N=16384 group 128", [(18432, 16384, 128, [16])], 2),
}

# grouped expert GEMM sweep: (description, experts, top-k, K, N, groupsize, [tokens ...])
MOE_CONFIGS = [
    ("8 experts top-2, K=4096 N=14336 (Mixtral-style expert up-projection)", 8, 2, 4096, 14336, 128, [1, 4, 16, 64, 256]),
    ("128 experts top-8, K=2048 N=1536 (Qwen3-30B-A3B-style fused gate/up)", 128, 8, 2048, 1536, 128, [1, 16, 64]),
    ("256 experts top-8, K=7168 N=4096 (DeepSeek-V3-style fused gate/up)", 256, 8, 7168, 4096, 128, [1, 16, 64]),
]

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


ZERO_POINTS = False  # set from --zero-points: the GEMM also reads a zero code per scale and a bias per column


def gemm_bytes(M, K, N, G):
    G = K if G in (-1, K) else G
    extra = (K // G) * N + 2 * N if ZERO_POINTS else 0
    return 2 * M * K + K * N // 2 + 2 * (K // G) * N + 2 * M * N + extra


def gemm_flops(M, K, N):
    return 2 * M * K * N


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return dict(FALLBACK_PEAKS, source="fallback")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="big")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph timing of layers under 20 us")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--only-m", type=int, default=None, help="run only this M of the sweep (profiling)")
    ap.add_argument("--no-cublas", action="store_true", help="skip the cuBLAS FP16 GEMM on the dequantised weights")
    ap.add_argument("--no-offline", action="store_true", help="skip timing the offline repack / quantise steps")
    ap.add_argument("--no-moe", action="store_true", help="skip the grouped expert (MoE) GEMM sweep")
    ap.add_argument("--no-ablation", action="store_true", help="skip the Figure 12 ablation sweep")
    ap.add_argument("--no-sparse", action="store_true", help="skip the 2:4-sparse GEMM sweep")
    ap.add_argument("--no-prefill", action="store_true", help="skip the compute-bound prefill layer")
    ap.add_argument("--min-reps", type=int, default=50,
                    help="launches per GEMM in the per-M statistics (200 below 10 us); fewer only for profiling")
    ap.add_argument("--moe-config", type=int, default=None, help="run only this entry of the MoE sweep (profiling)")
    ap.add_argument("--no-per-expert", action="store_true",
                    help="skip the one-launch-per-expert comparison of the MoE sweep (profiling)")
    ap.add_argument("--zero-points", action="store_true",
                    help="run every GEMM with a zero point per group and a bias (w4a16_gemm_zp)")
    ap.add_argument("--cpu-sample", default=None, help=argparse.SUPPRESS)  # internal: oracle timing child
    return ap.parse_args()


# ---------------------------------------------------------------------------
# CPU oracle timing (the cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def _oracle_gemm_blocks(A, q, s, G, cores, block=512):
    """The oracle's GEMM over the columns of (q, s), run as independent column blocks on
    `cores` threads (numpy releases the GIL inside its array kernels; BLAS is kept
    single-threaded per block).  The oracle itself is called as it stands."""
    from concurrent.futures import ThreadPoolExecutor
    import numpy as np
    import oracle
    N = q.shape[1]
    spans = [(c0, min(N, c0 + block)) for c0 in range(0, N, block)]

    def one(span):
        c0, c1 = span
        oracle.gemm_ref(A, np.ascontiguousarray(q[:, c0:c1]), np.ascontiguousarray(s[:, c0:c1]), G)

    with ThreadPoolExecutor(max_workers=cores) as ex:
        list(ex.map(one, spans))


def _cpu_sample_child(spec: str):
    """Time the oracle on a column sample of every GEMM of the workload (runs in a child
    process, threaded over column blocks on `cores` host threads); prints JSON
    {seconds, scaled_seconds, sample, cores, extrapolated}."""
    import numpy as np
    import oracle
    from mixed_precision_w4a16_gb300 import synth
    workload, ncols, cores, *opts = spec.split(":")
    ncols, cores = int(ncols), int(cores)
    time_repack = "repack" in opts
    desc, layers, seed = WORKLOADS[workload]
    total = 0.0
    scaled = 0.0
    repack = None
    extrapolated = False
    for li, (K, N, G, Ms) in enumerate(layers):
        nc = min(ncols, N)
        extrapolated |= nc < N
        q, s = synth.make_weights(K, nc, G, seed * 100 + li)  # same distributions, sample width
        if li == 0 and time_repack:  # the offline repack of the first layer, on its first REPACK_SAMPLE_COLS columns
            nr = min(REPACK_SAMPLE_COLS, nc)
            qr, sr = np.ascontiguousarray(q[:, :nr]), np.ascontiguousarray(s[:, :nr])
            t0 = time.perf_counter()
            oracle.repack(qr, sr, G)
            dt = time.perf_counter() - t0
            repack = {"seconds": dt, "scaled_seconds": dt * (N / nr), "shape": f"K={K} N={N} G={G}",
                      "sample": f"{nr} of its N columns, one thread, time scaled by N/cols"}
        for M in Ms:
            A = synth.make_activations(M, K, seed * 1000 + M)
            t0 = time.perf_counter()
            _oracle_gemm_blocks(A, q, s, G, cores)
            dt = time.perf_counter() - t0
            total += dt
            scaled += dt * (N / nc)
    how = f"threaded over 512-column blocks on {cores} host threads"
    sample = (f"every GEMM of the workload on {ncols} of its N columns, {how}; time extrapolated by N/cols"
              if extrapolated else f"every GEMM of the workload on all its columns, {how}")
    print(json.dumps({"seconds": total, "scaled_seconds": scaled, "repack": repack, "cores": cores,
                      "extrapolated": extrapolated, "sample": sample}))


def host_cores():
    """Host threads the oracle timing uses: every core this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_cpu_sample(workload: str, ncols: int, repack: bool = False, cores: int | None = None):
    cores = cores or host_cores()
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    spec = f"{workload}:{ncols}:{cores}" + (":repack" if repack else "")
    out = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-sample", spec],
                         capture_output=True, text=True, env=env, timeout=900)
    if out.returncode != 0:
        raise RuntimeError(f"oracle timing failed: {out.stderr[-2000:]}")
    return json.loads(out.stdout.strip().splitlines()[-1])


def workload_totals(layers):
    tb = sum(gemm_bytes(M, K, N, G) for K, N, G, Ms in layers for M in Ms)
    tf = sum(gemm_flops(M, K, N) for K, N, G, Ms in layers for M in Ms)
    return tb, tf


def cpu_sample_cols(workload, cores=1):
    """Columns of each GEMM the oracle computes for the cpu_baseline leg: about 10-20 s of wall
    time with `cores` threads (the per-thread figure was measured single-threaded), in whole
    512-column blocks."""
    per_core = {"big": 12288, "pr1": 1024, "7b": 16384, "70b": 8192, "prefill": 2048,
                "profile_m32": 4096, "profile_m8": 4096, "profile_m16": 4096}[workload]
    return max(512, per_core * max(1, cores) // 512 * 512)


# the files that decide what the GEMM kernels execute and how the work is split
GEMM_SOURCES = ("common.cuh", "gemm_launch.cu", "gemm_mma.cu", "gemm_tc.cu", "internal.h")


def _code_only(text):
    """C++ source without comments and with whitespace runs collapsed: what decides the build."""
    import re
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"' or c == "'":  # string or character literal, copied whole
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return re.sub(r"\s+", " ", "".join(out)).strip()


def kernel_source_hash(sources=None):
    """Hash of the GEMM kernels' code and their work planning (comments and layout excluded);
    profile figures are used only for the build they were taken on.  `sources` maps file name to
    text (default: the files in csrc/)."""
    import hashlib
    h = hashlib.sha256()
    for name in GEMM_SOURCES:
        h.update(name.encode())
        if sources is not None:
            text = sources[name]
        else:
            with open(os.path.join(ROOT, "mixed_precision_w4a16_gb300", "csrc", name), encoding="utf-8") as f:
                text = f.read()
        h.update(_code_only(text).encode())
    return h.hexdigest()[:16]


def profiled_traffic(name):
    """Per-launch DRAM bytes {(kernel, M, launch): bytes} from a committed ncu summary, or None when
    the summary was taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", name)
    try:
        with open(path) as f:
            text = f.read()
    except OSError:
        return None
    if f"kernel-source: {kernel_source_hash()}" not in text:
        return None
    out = {}
    for line in text.splitlines():
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) == 9 and cells[0].startswith("gemm_") and cells[1].isdigit():
            out[(cells[0], int(cells[1]), int(cells[2]))] = float(cells[6]) * 1e6
    return out or None


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi sampled every 100 ms on a reader thread; samples are time-stamped so
    that only those taken inside the timed region are summarised."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, uuid):
        import threading
        self.samples = []
        self.t_start = self.t_end = None
        self.static = self.read_once(uuid)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if uuid:
            cmd += ["-i", uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    @staticmethod
    def read_once(uuid):
        """Memory clock (current, max) and ECC mode, read once before the timed region; {} if
        nvidia-smi cannot tell."""
        cmd = ["nvidia-smi", "--query-gpu=clocks.mem,clocks.max.mem,ecc.mode.current", "--format=csv,noheader,nounits"]
        if uuid:
            cmd += ["-i", uuid]
        try:
            out = subprocess.run(cmd, capture_output=True, text=True, timeout=20)
            parts = [p.strip() for p in out.stdout.strip().splitlines()[0].split(",")]
        except Exception:
            return {}
        if out.returncode != 0 or len(parts) != 3:
            return {}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        return {"mem_mhz": num(parts[0]), "mem_max_mhz": num(parts[1]), "ecc": parts[2]}

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def start_timing(self):
        self.t_start = time.time()

    def stop_timing(self):
        self.t_end = time.time()

    def finish(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0,
                    **self.static}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        inside = [p for t, p in self.samples if self.t_start is not None and self.t_start <= t <= (self.t_end or t)]
        note = "samples inside the timed region"
        if not inside:  # timed region shorter than one sampling period: take the nearest samples
            near = sorted(self.samples, key=lambda tp: abs(tp[0] - (self.t_start or tp[0])))[:3]
            inside = [p for _, p in near]
            note = "nearest samples (timed region shorter than the sampling period)"

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [v for v in (num(p[1]) for p in inside) if v is not None]
        smax = [v for v in (num(p[2]) for p in inside) if v is not None]
        power = [v for v in (num(p[3]) for p in inside) if v is not None]
        reasons = sorted({name for p in inside for name, v in zip(self.REASONS, p[5:9])
                          if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(inside), "power_w_max": max(power) if power else None,
                "note": note, **self.static}


class NvmlClockSampler:
    """SM clock, power and clock-event reasons read through NVML (libnvidia-ml, by ctypes) every
    2 ms on a reader thread, so that even a timed region of a few tens of milliseconds holds
    several samples.  Only reads: no setting of the GPU is touched.  Raises OSError when NVML
    cannot be loaded or the GPU not found (the nvidia-smi sampler is used then)."""
    PERIOD_S = 0.002
    # clock-event reason bits of NVML's public header (nvmlClocksEventReason*)
    REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                   "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}

    def __init__(self, uuid):
        import ctypes
        import threading
        self.samples = []
        self.t_start = self.t_end = None
        self.static = ClockSampler.read_once(uuid)
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.lib = lib
        self.dev = ctypes.c_void_p()
        if not uuid or lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.dev)) != 0:
            raise OSError("GPU not found by UUID")
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        mx = ctypes.c_uint()
        self.sm_max = float(mx.value) if lib.nvmlDeviceGetMaxClockInfo(self.dev, 1, ctypes.byref(mx)) == 0 else None
        self.stop = False
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        import ctypes
        clk, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop:
            t = time.time()
            ok = self.lib.nvmlDeviceGetClockInfo(self.dev, 1, ctypes.byref(clk)) == 0  # NVML_CLOCK_SM
            p = pw.value / 1000.0 if self.lib.nvmlDeviceGetPowerUsage(self.dev, ctypes.byref(pw)) == 0 else None
            r = rs.value if self.reasons_fn(self.dev, ctypes.byref(rs)) == 0 else 0
            if ok:
                self.samples.append((t, float(clk.value), p, r))
            time.sleep(self.PERIOD_S)

    def start_timing(self):
        self.t_start = time.time()

    def stop_timing(self):
        self.t_end = time.time()

    def finish(self):
        self.stop = True
        self.thread.join(timeout=2)
        try:
            self.lib.nvmlShutdown()
        except Exception:
            pass
        inside = [x for x in self.samples if self.t_start is not None and self.t_start <= x[0] <= (self.t_end or x[0])]
        note = f"NVML samples every {self.PERIOD_S * 1e3:.0f} ms inside the timed region"
        if not inside:
            inside = sorted(self.samples, key=lambda x: abs(x[0] - (self.t_start or x[0])))[:3]
            note = "nearest NVML samples (none inside the timed region)"
        sm = [x[1] for x in inside]
        power = [x[2] for x in inside if x[2] is not None]
        reasons = sorted({name for x in inside for name, bit in self.REASON_BITS.items() if x[3] & bit})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.sm_max, "reasons": reasons,
                "samples": len(inside), "power_w_max": max(power) if power else None, "note": note, **self.static}


def make_clock_sampler(uuid):
    try:
        return NvmlClockSampler(uuid)
    except Exception:
        return ClockSampler(uuid)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args, rank, world, device):
    import numpy as np
    import torch
    import mixed_precision_w4a16_gb300 as w
    from mixed_precision_w4a16_gb300 import build, synth

    build.build()
    desc, layers, seed = WORKLOADS[args.workload]
    global ZERO_POINTS
    ZERO_POINTS = bool(args.zero_points)
    if args.only_m is not None:
        layers = [(K, N, G, [M for M in Ms if M == args.only_m]) for K, N, G, Ms in layers]
        layers = [l for l in layers if l[3]]
        if not layers:
            raise SystemExit(f"M={args.only_m} is not part of workload {args.workload}")
        desc += f" (only M={args.only_m})"
    peaks = load_peaks()
    stream = torch.cuda.current_stream()

    offline = None
    peaks_for_offline = load_peaks()
    # ---- inputs: seeded synthetic weights -> device repack; activations resident in HBM
    points = []  # (K, N, G, M, [packed copies], sp copies, A_d, C_d)
    max_ws = 0
    for li, (K, N, G, Ms) in enumerate(layers):
        q, s = synth.make_weights(K, N, G, seed * 100 + li)
        q_d = torch.from_numpy(q).to(device)
        s_d = torch.from_numpy(s).to(device)
        del q
        lbytes = K * N // 2
        copies = max(1, math.ceil(3 * L2_BYTES / lbytes)) if lbytes < 2 * L2_BYTES else 1
        packs = [w.repack(q_d, s_d, G) for _ in range(copies)]
        zp_d = bias_d = None
        if args.zero_points:
            rng_z = np.random.default_rng(seed * 100 + li + 7)
            NG = q_d.shape[0] // synth.effective_group(K, G)
            zp_d = w.repack_zeros(torch.from_numpy(rng_z.integers(0, 16, (NG, N)).astype(np.uint8)).to(device), K, G)
            bias_d = torch.from_numpy(rng_z.normal(0, 1.0, N).astype(np.float16)).to(device)
        if li == 0 and rank == 0 and not args.no_offline:
            offline = time_offline_steps(w, torch, q_d, s_d, K, N, G, seed, peaks_for_offline)
        del q_d, s_d
        for M in Ms:
            A = synth.make_activations(M, K, seed * 1000 + M)
            A_d = torch.from_numpy(A).to(device)
            C_d = torch.empty((M, N), dtype=torch.float16, device=device)
            points.append({"K": K, "N": N, "G": G, "M": M, "packs": packs, "A": A, "A_d": A_d, "C_d": C_d,
                           "zp": zp_d, "bias": bias_d})
            max_ws = max(max_ws, w.w4a16_workspace_bytes(M, K, N, G))
    ws = torch.zeros(max_ws, dtype=torch.uint8, device=device)
    torch.cuda.synchronize()
    launches_per_step = 0
    for p in points:
        plan = w.w4a16_plan(p["M"], p["K"], p["N"], p["G"])
        p["launches"] = math.ceil(p["M"] / plan["m_chunk"])
        p["kernel"] = KERNEL_OF_PATH[plan["path"]]
        launches_per_step += p["launches"]

    def gemm_call(p, packed, sp):
        if args.zero_points:
            w.w4a16_gemm_zp(p["A_d"], packed, sp, p["zp"], p["bias"], p["C_d"], p["M"], p["K"], p["N"], p["G"], ws,
                            max_ws, stream)
        else:
            w.w4a16_gemm(p["A_d"], packed, sp, p["C_d"], p["M"], p["K"], p["N"], p["G"], ws, max_ws, stream)

    def one_step(it):
        for p in points:
            packed, sp = p["packs"][it % len(p["packs"])]
            gemm_call(p, packed, sp)

    for it in range(args.warmup):
        one_step(it)
    torch.cuda.synchronize()
    if w.w4a16_get_status(ws) != 0:
        raise RuntimeError("device status error during warm-up")

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        pass
    sampler = make_clock_sampler(uuid) if rank == 0 else None
    time.sleep(0.3)

    # ---- timed region: barrier + sync on both sides, CUDA events on the launching stream.  The
    # GEMMs of a step run back to back (no events between them, which would keep a kernel's
    # set-up from overlapping the previous one's tail); per-GEMM times come from the loop below.
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start_timing()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for it in range(args.steps):
        one_step(it)
    ev1.record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.stop_timing()
    if world > 1:
        torch.distributed.barrier()
    ms_total = ev0.elapsed_time(ev1)
    status = w.w4a16_get_status(ws)
    if status != 0:
        raise RuntimeError(f"device status error in timed region: {w.w4a16_status_string(status)}")

    # ---- end-to-end through the public API: pinned host A in, host C out, every step.  The
    # copies run on two copy streams next to the GEMMs' stream: a GEMM's input copy is issued
    # ahead and its output read starts as soon as it finishes, so copies overlap the other GEMMs.
    # Events keep every buffer in order: A_d[i] is refilled only after the previous step's GEMM i
    # read it, and GEMM i writes C_d[i] only after the previous step's read of it finished.
    e2e = None
    if not args.no_e2e:
        hostA = [torch.from_numpy(p["A"]).pin_memory() for p in points]
        hostC = [torch.empty(p["C_d"].shape, dtype=torch.float16).pin_memory() for p in points]
        h2d = sum(p["M"] * p["K"] * 2 for p in points)
        d2h = sum(p["M"] * p["N"] * 2 for p in points)
        e_steps = max(1, min(args.steps, 50))
        s_in = torch.cuda.Stream(device)
        s_out = torch.cuda.Stream(device)
        in_done = [torch.cuda.Event() for _ in points]
        gemm_done = [torch.cuda.Event() for _ in points]
        out_done = [torch.cuda.Event() for _ in points]

        def e2e_step(it, first):
            for i, p in enumerate(points):
                if not first:
                    s_in.wait_event(gemm_done[i])
                with torch.cuda.stream(s_in):
                    p["A_d"].copy_(hostA[i], non_blocking=True)
                in_done[i].record(s_in)
                stream.wait_event(in_done[i])
                if not first:
                    stream.wait_event(out_done[i])
                packed, sp = p["packs"][it % len(p["packs"])]
                gemm_call(p, packed, sp)
                gemm_done[i].record(stream)
                s_out.wait_event(gemm_done[i])
                with torch.cuda.stream(s_out):
                    hostC[i].copy_(p["C_d"], non_blocking=True)
                out_done[i].record(s_out)

        for it in range(2):
            e2e_step(it, it == 0)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        s_in.wait_event(e0)  # no copy of the timed steps starts before the timed region
        for it in range(e_steps):
            e2e_step(it, False)
        stream.wait_event(out_done[-1])  # the last read of C (the read stream runs in order)
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = e0.elapsed_time(e1) / e_steps
        e_ms = reduce_max(e_ms, world, device)
        tb, _ = workload_totals(layers)
        e2e = {"value": world * tb / (e_ms * 1e-3) / 1e12, "unit": "TB/s", "ms_per_step": e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e_steps,
               "copies": "H2D and D2H on two copy streams, overlapped with the GEMMs"}

    # ---- per-M statistics: a dedicated loop of at least 50 launches per GEMM (200 when its
    # roofline time is under 10 us), cycling through the L2-rotation copies, one event pair each
    rep_us = [[] for _ in points]
    if rank == 0:
        for i, p in enumerate(points):
            t_roof = max(gemm_bytes(p["M"], p["K"], p["N"], p["G"]) / (peaks["hbm_gbs"] * 1e9),
                         gemm_flops(p["M"], p["K"], p["N"]) / (peaks["bf16_tflops"] * 1e12))
            reps = max(args.steps, 4 * args.min_reps if t_roof < 10e-6 else args.min_reps)
            pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
            for it, (a, b) in enumerate(pairs):
                packed, sp = p["packs"][it % len(p["packs"])]
                a.record(stream)
                gemm_call(p, packed, sp)
                b.record(stream)
            torch.cuda.synchronize()
            rep_us[i] = [a.elapsed_time(b) for a, b in pairs]
        if w.w4a16_get_status(ws) != 0:
            raise RuntimeError("device status error in the per-M timing")

    # ---- context: cuBLAS FP16 GEMM (FP32 accumulation) on the dequantised weights, same A
    cublas_us = None
    if not args.no_cublas and rank == 0:
        torch.backends.cuda.matmul.allow_fp16_reduced_precision_reduction = False
        cublas_us = []
        bhat_cache = {}
        for p in points:
            key = (p["K"], p["N"], p["G"], id(p["packs"]))
            if key not in bhat_cache:
                bhat_cache.clear()
                packed, sp = p["packs"][0]
                bhat_cache[key] = w.dequant(packed, sp, p["K"], p["N"], p["G"])
            bhat = bhat_cache[key]
            out = torch.empty_like(p["C_d"])
            for _ in range(3):
                torch.matmul(p["A_d"], bhat, out=out)
            reps = 10
            c0 = torch.cuda.Event(enable_timing=True)
            c1 = torch.cuda.Event(enable_timing=True)
            c0.record(stream)
            for _ in range(reps):
                torch.matmul(p["A_d"], bhat, out=out)
            c1.record(stream)
            torch.cuda.synchronize()
            cublas_us.append(c0.elapsed_time(c1) / reps * 1e3)
        bhat_cache.clear()

    # ---- layers whose roofline time is under GRAPH_BELOW_US: time per GEMM inside a CUDA graph of
    # many launches as well (launch overhead amortised), next to the single-launch figure above
    graph_us = {}
    if rank == 0 and not args.no_graph:
        def graph_gemm(p, packed, sp):  # on the current (capturing) stream
            if args.zero_points:
                w.w4a16_gemm_zp(p["A_d"], packed, sp, p["zp"], p["bias"], p["C_d"], p["M"], p["K"], p["N"], p["G"],
                                ws, max_ws)
            else:
                w.w4a16_gemm(p["A_d"], packed, sp, p["C_d"], p["M"], p["K"], p["N"], p["G"], ws, max_ws)

        for i, p in enumerate(points):
            t_roof = max(gemm_bytes(p["M"], p["K"], p["N"], p["G"]) / (peaks["hbm_gbs"] * 1e9),
                         gemm_flops(p["M"], p["K"], p["N"]) / (peaks["bf16_tflops"] * 1e12))
            if t_roof * 1e6 >= GRAPH_BELOW_US:
                continue
            nl = max(GRAPH_LAUNCHES, len(p["packs"]))  # every L2-rotation copy once per replay
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for k in range(nl):
                    packed, sp = p["packs"][k % len(p["packs"])]
                    graph_gemm(p, packed, sp)
            g.replay()
            torch.cuda.synchronize()
            reps = 20
            g0 = torch.cuda.Event(enable_timing=True)
            g1 = torch.cuda.Event(enable_timing=True)
            g0.record(stream)
            for _ in range(reps):
                g.replay()
            g1.record(stream)
            torch.cuda.synchronize()
            graph_us[i] = (g0.elapsed_time(g1) / (reps * nl) * 1e3, nl)
            del g
        if graph_us and w.w4a16_get_status(ws) != 0:
            raise RuntimeError("device status error in the CUDA-graph timing")

    ms_per_step = reduce_max(ms_total / args.steps, world, device)
    clocks = sampler.finish() if sampler else None
    if rank != 0:
        return None

    tb, tf = workload_totals(layers)
    value = world * tb / (ms_per_step * 1e-3) / 1e12
    bw = peaks["hbm_gbs"] * 1e9
    pk = peaks["bf16_tflops"] * 1e12  # dense FP16 equals dense BF16 on this part
    sweep = []
    for p, ts in zip(points, rep_us):
        us = statistics.median(ts) * 1e3
        by = gemm_bytes(p["M"], p["K"], p["N"], p["G"])
        fl = gemm_flops(p["M"], p["K"], p["N"])
        t_roof = max(by / bw, fl / pk)
        mem_bound = by / bw >= fl / pk
        sweep.append({"M": p["M"], "K": p["K"], "N": p["N"], "group": p["G"], "us": round(us, 2),
                      "us_p10": round(sorted(ts)[len(ts) // 10] * 1e3, 2),
                      "us_p90": round(sorted(ts)[(9 * len(ts)) // 10] * 1e3, 2),
                      "tb_s": round(by / (us * 1e-6) / 1e12, 3), "tflops": round(fl / (us * 1e-6) / 1e12, 1),
                      "roofline_frac": round(t_roof / (us * 1e-6), 3), "bound": "hbm" if mem_bound else "tensor",
                      "launches": p["launches"], "kernel": p["kernel"], "reps": len(ts)})
        if len(sweep) - 1 in graph_us:
            gus, nl = graph_us[len(sweep) - 1]
            sweep[-1]["graph_us"] = round(gus, 2)
            sweep[-1]["graph_launches"] = nl
            sweep[-1]["graph_roofline_frac"] = round(t_roof / (gus * 1e-6), 3)
        if cublas_us is not None:
            cu = cublas_us[len(sweep) - 1]
            sweep[-1]["cublas_fp16_us"] = round(cu, 2)
            sweep[-1]["speedup_vs_cublas"] = round(cu / us, 3)
    roofline_by_kernel = []
    for kname in sorted({p["kernel"] for p in points}):
        rows = [(p, r) for p, r in zip(points, sweep) if p["kernel"] == kname]
        t_all = sum(r["us"] for _, r in rows)
        mem = [(p, r) for p, r in rows if r["bound"] == "hbm"]
        ten = [(p, r) for p, r in rows if r["bound"] == "tensor"]
        entry = {"kernel": kname, "us_per_step": round(t_all, 2), "points": [r["M"] for _, r in rows]}
        if mem:
            by = sum(gemm_bytes(p["M"], p["K"], p["N"], p["G"]) for p, _ in mem)
            t = sum(r["us"] for _, r in mem) * 1e-6
            nl = sum(p["launches"] for p, _ in mem)
            entry["hbm"] = {"achieved": round(by / t / 1e9, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                            "frac": round(by / t / 1e9 / peaks["hbm_gbs"], 3), "points": [r["M"] for _, r in mem],
                            "algorithmic_bytes_per_launch": round(by / nl), "launches": nl}
        if ten:
            fl = sum(gemm_flops(p["M"], p["K"], p["N"]) for p, _ in ten)
            t = sum(r["us"] for _, r in ten) * 1e-6
            entry["tensor"] = {"achieved": round(fl / t / 1e12, 1), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                               "frac": round(fl / t / 1e12 / peaks["bf16_tflops"], 3),
                               "points": [r["M"] for _, r in ten]}
        roofline_by_kernel.append(entry)
    # the dominant kernel: the largest share of the step's device time
    dom = max(roofline_by_kernel, key=lambda e: e["us_per_step"])
    prof = profiled_traffic("gemm_big_layer_traffic.md") if args.workload == "big" else None
    if "hbm" in dom:
        traffic = None
        if prof:
            vals = [v for (k, m, _), v in prof.items() if k == dom["kernel"] and m in dom["hbm"]["points"]]
            if vals:
                traffic = round(sum(vals) / len(vals))
        h = dom["hbm"]
        roofline = {"bound": "hbm", "achieved": h["achieved"], "peak": h["peak"], "unit": "GB/s",
                    "frac": h["frac"], "traffic": traffic,
                    "algorithmic_bytes_per_launch": h["algorithmic_bytes_per_launch"],
                    "kernel": dom["kernel"], "over": f"its memory-bound points M={h['points']}",
                    "share_of_step": round(dom["us_per_step"] / sum(e["us_per_step"] for e in roofline_by_kernel), 3),
                    "peak_source": peaks["source"]}
    else:
        t = dom["tensor"]
        roofline = {"bound": "tensor", "achieved": t["achieved"], "peak": t["peak"], "unit": "TFLOP/s",
                    "frac": t["frac"], "traffic": None, "kernel": dom["kernel"],
                    "over": f"its points M={t['points']}", "peak_source": peaks["source"]}

    moe = None
    if rank == 0 and not args.no_moe and args.workload == "big":
        moe = time_moe(w, torch, device, peaks, args.moe_config, not args.no_per_expert)
    ablation = None
    if rank == 0 and not args.no_ablation and args.workload == "big" and not args.zero_points:
        ablation = time_ablations(w, torch, points, ws, max_ws, stream)
    sparse24 = None
    if rank == 0 and not args.no_sparse and args.workload == "big" and not args.zero_points:
        sparse24 = time_sparse24(w, torch, device, peaks, {r["M"]: r["us"] for r in sweep})

    prefill = None
    if rank == 0 and not args.no_prefill and args.workload == "big" and not args.zero_points:
        prefill = time_prefill(w, torch, device, peaks, stream, not args.no_cublas, args.min_reps)

    cpu = None
    if not args.no_cpu_baseline:
        cores = host_cores()
        ncols = cpu_sample_cols(args.workload, cores)
        r = run_cpu_sample(args.workload, ncols, repack=True, cores=cores)
        cpu = {"value": tb / r["scaled_seconds"] / 1e12, "unit": "TB/s", "cores": r["cores"], "kind": "oracle",
               "extrapolated": r["extrapolated"],
               "sample": r["sample"] + f"; measured {r['seconds']:.1f} s wall"}
        if r.get("repack"):
            cpu["oracle_repack_us"] = round(r["repack"]["scaled_seconds"] * 1e6, 1)
            cpu["oracle_repack_sample"] = f"{r['repack']['shape']}, {r['repack']['sample']}"

    return {
        "metric": METRIC, "value": round(value, 4), "unit": "TB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": desc, "gemms_per_step": len(points),
                   "l2": "inputs larger than L2" if all(len(p["packs"]) == 1 for p in points)
                   else "weight copies rotated to exceed 3x L2",
                   "parallelism": f"replicas x{world}", "peaks": peaks["source"],
                   "variant": "zero point per group + bias" if args.zero_points else "symmetric (z = 8)"},
        "sweep": sweep, "roofline": roofline, "roofline_by_kernel": roofline_by_kernel,
        "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps, "clocks": clocks, "offline": offline,
        "moe": moe, "ablation": ablation, "sparse24": sparse24, "prefill": prefill,
    }


PREFILL = (8192, 28672, 128, (256, 512, 1024))


def time_prefill(w, torch, device, peaks, stream, with_cublas=True, min_reps=50):
    """The compute-bound prefill layer (K=8192, N=28672, group 128, M in {256, 512, 1024}),
    outside the timed region: per M the median of 50 launches, cycling through weight copies
    that together exceed 3x L2 (one copy, 117 MB, would fit), against the dense FP16 tensor peak
    (the measured cuBLAS BF16 figure: FP16 and BF16 have the same dense rate).  For context, a
    cuBLAS FP16 GEMM (FP32 accumulation) on the dequantised weights."""
    import numpy as np
    from mixed_precision_w4a16_gb300 import synth
    K, N, G, Ms = PREFILL
    q, s = synth.make_weights(K, N, G, 400)
    q_d, s_d = torch.from_numpy(q).to(device), torch.from_numpy(s).to(device)
    del q
    copies = max(1, math.ceil(3 * L2_BYTES / (K * N // 2)))
    packs = [w.repack(q_d, s_d, G) for _ in range(copies)]
    del q_d, s_d
    bhat = w.dequant(packs[0][0], packs[0][1], K, N, G) if with_cublas else None
    out = []
    for M in Ms:
        A_d = torch.from_numpy(synth.make_activations(M, K, 400 * 1000 + M)).to(device)
        C_d = torch.empty((M, N), dtype=torch.float16, device=device)
        ws_bytes = w.w4a16_workspace_bytes(M, K, N, G)
        ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=device)
        plan = w.w4a16_plan(M, K, N, G)
        for it in range(3):
            packed, sp = packs[it % copies]
            w.w4a16_gemm(A_d, packed, sp, C_d, M, K, N, G, ws, ws_bytes, stream)
        reps = max(1, min_reps)
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for it, (a, b) in enumerate(pairs):
            packed, sp = packs[it % copies]
            a.record(stream)
            w.w4a16_gemm(A_d, packed, sp, C_d, M, K, N, G, ws, ws_bytes, stream)
            b.record(stream)
        torch.cuda.synchronize()
        ts = sorted(a.elapsed_time(b) * 1e3 for a, b in pairs)
        if w.w4a16_get_status(ws) != 0:
            raise RuntimeError("device status error in the prefill timing")
        us = statistics.median(ts)
        fl = gemm_flops(M, K, N)
        by = gemm_bytes(M, K, N, G)
        tflops = fl / (us * 1e-6) / 1e12
        t_roof = max(by / (peaks["hbm_gbs"] * 1e9), fl / (peaks["bf16_tflops"] * 1e12))
        entry = {"M": M, "K": K, "N": N, "group": G, "us": round(us, 2), "us_p10": round(ts[reps // 10], 2),
                 "us_p90": round(ts[min(reps - 1, (9 * reps) // 10)], 2), "reps": reps, "tflops": round(tflops, 1),
                 "frac_of_tensor_peak": round(tflops / peaks["bf16_tflops"], 3),
                 "frac_of_sustained_tensor_peak": round(tflops / peaks["bf16_tflops_sustained"], 3),
                 "roofline_frac": round(t_roof / (us * 1e-6), 3), "bytes": by,
                 "launches": math.ceil(M / plan["m_chunk"]), "kernel": KERNEL_OF_PATH[plan["path"]]}
        if bhat is not None:
            c = torch.empty((M, N), dtype=torch.float16, device=device)
            for _ in range(3):
                torch.matmul(A_d, bhat, out=c)
            c0 = torch.cuda.Event(enable_timing=True)
            c1 = torch.cuda.Event(enable_timing=True)
            c0.record(stream)
            for _ in range(10):
                torch.matmul(A_d, bhat, out=c)
            c1.record(stream)
            torch.cuda.synchronize()
            cu = c0.elapsed_time(c1) / 10 * 1e3
            entry["cublas_fp16_us"] = round(cu, 2)
            entry["cublas_fp16_tflops"] = round(fl / (cu * 1e-6) / 1e12, 1)
            entry["speedup_vs_cublas"] = round(cu / us, 3)
            del c
        out.append(entry)
        del A_d, C_d, ws
    del packs, bhat
    return {"peak": peaks["bf16_tflops"], "peak_sustained": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
            "peak_source": peaks["source"], "l2": f"{copies} weight copies rotated (> 3x L2)", "points": out}


def gemm24_bytes(M, K, N, G):
    """Algorithmic bytes of the 2:4-sparse GEMM: 3 bits per weight (two 4-bit codes and two
    2-bit positions per group of four) instead of 4."""
    G = K if G in (-1, K) else G
    return 2 * M * K + 3 * K * N // 8 + 2 * (K // G) * N + 2 * M * N


def time_sparse24(w, torch, device, peaks, dense_us):
    """2:4-sparse GEMM on the big layer (outside the timed region): the packed stream is random
    codes with random rising position pairs (each of the six pairs equally likely), generated on
    the device; the weights (510 MB) exceed L2.  Compared with the dense GEMM of the sweep at the
    same M."""
    K, N, G = 18432, 73728, 128
    gen = torch.Generator(device=device)
    gen.manual_seed(13)
    packed = torch.randint(-2 ** 31, 2 ** 31, (3 * K * N // 32,), dtype=torch.int32, device=device, generator=gen)
    pieces = packed.view(-1, 768)                       # per 128-column strip and 64-row piece
    lut = torch.tensor([4, 8, 12, 9, 13, 14], dtype=torch.int64, device=device)  # rising pairs (i0 | i1 << 2)
    shifts = 4 * torch.arange(8, device=device, dtype=torch.int64)
    for c0 in range(0, pieces.shape[0], 16384):
        blk = pieces[c0:c0 + 16384]
        nib = lut[torch.randint(0, 6, (blk.shape[0], 256, 8), device=device, generator=gen)]
        meta = (nib << shifts).sum(-1)
        blk[:, 512:] = torch.where(meta >= 2 ** 31, meta - 2 ** 32, meta).to(torch.int32)
    del nib, meta
    sp = (torch.rand(K // G * N, device=device, generator=gen) * 0.018 + 0.002).to(torch.float16)
    out = []
    for M in (1, 8, 16, 32, 64):
        A_d = torch.randn(M, K, device=device, generator=gen).to(torch.float16)
        C_d = torch.empty((M, N), dtype=torch.float16, device=device)
        ws = torch.zeros(w.w4a16_workspace_bytes_24(M, K, N, G), dtype=torch.uint8, device=device)
        for _ in range(3):
            w.w4a16_gemm_24(A_d, packed, sp, C_d, M, K, N, G, ws)
        times = []
        for _ in range(20):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            w.w4a16_gemm_24(A_d, packed, sp, C_d, M, K, N, G, ws)
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3)
        us = statistics.median(times)
        nbytes = gemm24_bytes(M, K, N, G)
        gbs = nbytes / (us * 1e-6) / 1e9
        entry = {"M": M, "K": K, "N": N, "group": G, "us": round(us, 1), "bytes": nbytes, "gb_s": round(gbs, 1),
                 "roofline_frac": round(gbs / peaks["hbm_gbs"], 3)}
        if M in dense_us:
            entry["dense_us"] = dense_us[M]
            entry["speedup_vs_dense"] = round(dense_us[M] / us, 3)
        out.append(entry)
        if w.w4a16_get_status(ws) != 0:
            raise RuntimeError("device status error in the 2:4 sweep")
    del packed, sp
    return out


ABLATIONS = [("full design", 0), ("no evict-first on weights", 1), ("2 pipeline stages", 2),
             ("no activation swizzle", 4), ("all three", 7)]


def time_ablations(w, torch, points, ws, max_ws, stream):
    """The MARLIN paper's Figure 12 ablations re-run on this library's kernels (outside the timed
    region): per M of the sweep, the median device time of one GEMM with each switch of
    w4a16_debug_ablate, and the slowdown against the full design.  The no-swizzle switch applies
    to the streaming kernel only (M <= 16)."""
    out = {"variants": [name for name, _ in ABLATIONS], "points": []}
    try:
        for p in points:
            row = {"M": p["M"], "kernel": p["kernel"], "us": {}}
            for name, flags in ABLATIONS:
                w.w4a16_debug_ablate(flags)
                times = []
                for it in range(8):
                    packed, sp = p["packs"][it % len(p["packs"])]
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    w.w4a16_gemm(p["A_d"], packed, sp, p["C_d"], p["M"], p["K"], p["N"], p["G"], ws, max_ws, stream)
                    e1.record(stream)
                    torch.cuda.synchronize()
                    if it >= 2:
                        times.append(e0.elapsed_time(e1) * 1e3)
                row["us"][name] = round(statistics.median(times), 1)
            full = row["us"]["full design"]
            row["slowdown"] = {k: round(v / full, 3) for k, v in row["us"].items() if k != "full design"}
            out["points"].append(row)
    finally:
        w.w4a16_debug_ablate(0)
    if w.w4a16_get_status(ws) != 0:
        raise RuntimeError("device status error in the ablation sweep")
    return out


def time_moe(w, torch, device, peaks, only_config=None, per_expert_context=True):
    """Grouped expert GEMM (outside the timed region): one w4a16_moe_gemm over every expert of an
    MoE layer, for routed batches of a few sizes.  The weights are random packed words (random
    4-bit codes) and scales generated on the device; each timed call follows an L2 flush.  Bytes
    are algorithmic: each expert that owns rows read once, plus A and C.  For context, the same
    work as one w4a16_gemm launch per expert that owns rows."""
    import numpy as np
    from mixed_precision_w4a16_gb300 import synth
    gen = torch.Generator(device=device)
    gen.manual_seed(11)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)
    out = []
    for ci, (desc, E, topk, K, N, G, token_list) in enumerate(MOE_CONFIGS):
        if only_config is not None and ci != only_config:
            continue
        NG = K // synth.effective_group(K, G)
        wpe, spe = K * N // 8, NG * N
        packed = torch.randint(-2 ** 31, 2 ** 31, (E * wpe,), dtype=torch.int32, device=device, generator=gen)
        sp = (torch.rand(E * spe, device=device, generator=gen) * 0.018 + 0.002).to(torch.float16)
        for tokens in token_list:
            counts = synth.make_expert_rows(tokens, topk, E, seed=100 * ci + tokens)
            offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
            M = int(offsets[-1])
            max_rows = int(counts.max())
            A_d = torch.from_numpy(synth.make_activations(M, K, seed=7)).to(device)
            C_d = torch.empty((M, N), dtype=torch.float16, device=device)
            off_d = torch.from_numpy(offsets).to(device)
            ws = w.moe_workspace_for(E, M, max_rows, K, N, G, device)
            active = [e for e in range(E) if counts[e] > 0]
            dense_ws = torch.zeros(max(w.w4a16_workspace_bytes(int(counts[e]), K, N, G) for e in active),
                                   dtype=torch.uint8, device=device)

            def grouped():
                w.w4a16_moe_gemm(A_d, packed, sp, off_d, C_d, E, M, max_rows, K, N, G, ws)

            def per_expert():
                for e in active:
                    lo, hi = int(offsets[e]), int(offsets[e + 1])
                    w.w4a16_gemm(A_d[lo:hi], packed[e * wpe:(e + 1) * wpe], sp[e * spe:(e + 1) * spe], C_d[lo:hi],
                                 hi - lo, K, N, G, dense_ws)

            res = {"per_expert": None}
            for name, fn in (("grouped", grouped), ("per_expert", per_expert)):
                if name == "per_expert" and not per_expert_context:
                    continue
                for _ in range(3):
                    fn()
                times = []
                for _ in range(10):
                    flush.fill_(1)
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record()
                    fn()
                    e1.record()
                    torch.cuda.synchronize()
                    times.append(e0.elapsed_time(e1) * 1e3)
                res[name] = statistics.median(times)
            if w.w4a16_get_status(ws) != 0:
                raise RuntimeError("device status error in the grouped GEMM")
            nbytes = len(active) * (K * N // 2 + 2 * NG * N) + 2 * M * K + 2 * M * N
            gbs = nbytes / (res["grouped"] * 1e-6) / 1e9
            out.append({"config": desc, "tokens": tokens, "rows": M, "active_experts": len(active),
                        "max_rows_per_expert": max_rows,
                        "kernel": "gemm_tc_kernel" if max_rows >= 17 else "gemm_mma_kernel",  # the library's rule
                        "us": round(res["grouped"], 1), "bytes": nbytes,
                        "gb_s": round(gbs, 1), "roofline_frac": round(gbs / peaks["hbm_gbs"], 3),
                        "per_expert_launches_us": None if res["per_expert"] is None else round(res["per_expert"], 1)})
            del A_d, C_d, ws, dense_ws
        del packed, sp
    del flush
    return out


def time_offline_steps(w, torch, q_d, s_d, K, N, G, seed, peaks):
    """Device time of the offline steps on the first layer of the workload (outside the
    timed region): w4a16_repack (codes uint8 in, packed + permuted scales out),
    w4a16_quantize_repack (FP16 weights in) and w4a16_minmax_scales (FP16 weights in,
    scales and zero codes out), against the HBM roofline of the bytes each reads and writes once."""
    from mixed_precision_w4a16_gb300 import synth
    wt, s16 = synth.make_fp16_weights(K, N, G, seed)
    w_d = torch.from_numpy(wt).to(q_d.device)
    s2_d = torch.from_numpy(s16).to(q_d.device)
    del wt
    NG = K // synth.effective_group(K, G)
    out = {}
    packed_out = K * N // 2 + 2 * NG * N  # packed stream and permuted scales, written once
    for name, fn, nbytes in (
            ("repack", lambda: w.repack(q_d, s_d, G), K * N + 2 * NG * N + packed_out),
            ("quantize_repack", lambda: w.quantize_repack(w_d, s2_d, G), 2 * K * N + 2 * NG * N + packed_out),
            ("minmax_scales", lambda: w.minmax_scales(w_d, G, symmetric=False), 2 * K * N + 3 * NG * N)):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        reps = 5
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) / reps * 1e3
        out[name] = {"us": round(us, 1), "bytes": nbytes, "gb_s": round(nbytes / (us * 1e-6) / 1e9, 1),
                     "roofline_frac": round(nbytes / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 3),
                     "shape": f"K={K} N={N} G={G}"}
    if w.w4a16_get_status() != 0:
        raise RuntimeError("device status error in the offline steps")
    del w_d, s2_d
    return out


def reduce_max(x, world, device):
    """Max of a host number over all ranks (NCCL on GPUs, gloo on CPU)."""
    if world <= 1:
        return x
    import torch
    dist = torch.distributed
    dev = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle, timed as it stands on the host cores
# ---------------------------------------------------------------------------

def run_reference(args, rank, world):
    if rank != 0:
        return None
    desc, layers, seed = WORKLOADS[args.workload]
    tb, _ = workload_totals(layers)
    cores = host_cores()
    # a smaller sample than the cpu_baseline leg: every step re-runs it
    ncols = max(512, cpu_sample_cols(args.workload, cores) // 32 // 512 * 512)
    for _ in range(args.warmup):
        run_cpu_sample(args.workload, ncols, cores=cores)
    secs = []
    extrapolated = False
    t0 = time.perf_counter()
    for _ in range(args.steps):
        r = run_cpu_sample(args.workload, ncols, cores=cores)
        secs.append(r["scaled_seconds"])
        extrapolated |= r["extrapolated"]
    wall = time.perf_counter() - t0
    s_step = statistics.mean(secs)
    v = tb / s_step / 1e12
    how = (f"extrapolated from a column sample ({ncols} columns of each GEMM, time scaled by N/cols)"
           if extrapolated else "every column of each GEMM")
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": s_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": desc, "parallelism": f"single host process, {cores} threads",
                   "timing": how},
        "cpu_baseline": {"value": v, "unit": "TB/s", "cores": cores, "kind": "oracle", "extrapolated": extrapolated,
                         "sample": f"each step: every GEMM of the workload, {how}, threaded over 512-column "
                                   f"blocks (wall {wall:.1f} s for {args.steps} steps)"},
        "e2e": {"value": v, "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    if args.cpu_sample:
        _cpu_sample_child(args.cpu_sample)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    import torch
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=device)
    try:
        out = run_ours(args, rank, world, device)
        if out is not None:
            print(json.dumps(out), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
