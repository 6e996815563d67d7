"""Benchmark: skinny BF16 GEMM + fused residual on GB300.

Workload (the decode-sized latent-MoE projection of the vLLM
"benchmark_k3_cutedsl_residual.py" page): Y = bf16(A . W^T + R) with
N = 7168, K = 3584, for each M in {1, 2, 4, 8, 16}, with 4 rotating copies of
W (~205 MB together, more than the 136 MB L2 the device reports) so every call streams W from
HBM.  One step = one call per (M, copy) pair = 20 calls, captured once in a
CUDA graph and replayed (the page's graph-replay method).  Synthetic inputs:
A, R ~ N(0,1), W ~ N(0,1)/sqrt(K), BF16, seeded.

Prints ONE JSON line (rank 0).  `value` is achieved HBM GB/s over the whole
step: algorithmic bytes 2*(N*K + M*K + 2*M*N) per call, summed over the
step's calls, divided by the device time per step (CUDA events).  The timed
region of K steps is repeated until the repeats span about two seconds (so
that the clock sampler sees the load); `value` and `ms_per_step` come from
the median repeat, `headline` holds the spread.
Per-M microseconds per call (median of repeats, the page's summary) are in
`per_m`, with the cuBLAS `torch.addmm` comparator timed the same way beside
each M.  `transition` times every kernel path at M = 32, 64, 128 and
`compute_bound` the library's choice at M = 256, 512, 1024 against the BF16
tensor peak, both with the same comparator (the page's `addmm` backend and
`graph_samples` method).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (FP64 C loop) on the host cores on a
bounded sample of the same workload, as the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
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

METRIC = "µs/call and achieved HBM GB/s, BF16 skinny GEMM+residual, M=1..16, N7168 K3584"
N_DIM, K_DIM = 7168, 3584
M_LIST = (1, 2, 4, 8, 16)
COPIES = 4
PATH_NAMES = {1: "simt", 2: "tc", 3: "rows", 4: "tile", 6: "pair"}
PATH_IDS = {v: k for k, v in PATH_NAMES.items()}
TRANSITION_M = (32, 64, 128)
COMPUTE_M = (256, 512, 1024)
KERNEL_NAMES = {"simt": "simt_skinny_kernel", "tc": "tc_skinny_kernel", "rows": "rows_skinny_kernel",
                "tile": "tile_gemm_kernel", "pair": "pair_gemm_kernel"}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def set_shape(n: int, k: int) -> None:
    """Another projection shape (e.g. the down-projection, --n 3584 --k 7168):
    every leg runs on it and the metric names it."""
    global N_DIM, K_DIM, METRIC
    if (n, k) != (N_DIM, K_DIM):
        METRIC = METRIC.replace(f"N{N_DIM} K{K_DIM}", f"N{n} K{k}")
        N_DIM, K_DIM = n, k


def alg_bytes(M: int, N: int | None = None, K: int | None = None) -> int:
    N = N_DIM if N is None else N
    K = K_DIM if K is None else K
    return 2 * (N * K + M * K + 2 * M * N)


def alg_flops(M: int, N: int | None = None, K: int | None = None) -> int:
    N = N_DIM if N is None else N
    K = K_DIM if K is None else K
    return 2 * M * N * K


def tensor_bound(M: int, peaks: dict) -> bool:
    """True when the call's FLOPs at the BF16 tensor peak take longer than its
    bytes at the HBM peak (the roofline's ridge point lies below M)."""
    return alg_flops(M) / (peaks["bf16_tflops"] * 1e12) > alg_bytes(M) / (peaks["hbm_gbs"] * 1e9)


def workload_name(m_list) -> str:
    """The `config.workload` both arms report for the same M sweep."""
    return f"M sweep {list(m_list)} x {COPIES} rotating W/R copies, N={N_DIM}, K={K_DIM}"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"]))}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# Source files each kernel is compiled from: a committed DRAM-traffic figure
# stays valid while these files are unchanged.
KERNEL_SOURCES = {
    "simt_skinny_kernel": ("sgr_simt.cuh", "sgr_ptx.cuh"),
    "rows_skinny_kernel": ("sgr_rows.cuh", "sgr_epi.cuh", "sgr_tc.cuh", "sgr_ptx.cuh"),
    "tc_skinny_kernel": ("sgr_tc.cuh", "sgr_ptx.cuh"),
    "tile_gemm_kernel": ("sgr_gemm.cuh", "sgr_tc.cuh", "sgr_ptx.cuh"),
    "pair_gemm_kernel": ("sgr_pair.cuh", "sgr_gemm.cuh", "sgr_tc.cuh", "sgr_ptx.cuh"),
    "w8_rows_kernel": ("sgr_w8.cuh", "sgr_tc.cuh", "sgr_ptx.cuh"),
    "w8s_kernel": ("sgr_w8s.cuh", "sgr_epi.cuh", "sgr_w8.cuh", "sgr_tc.cuh", "sgr_ptx.cuh"),
}


def kernel_source_digest(kernel: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "skinny_bf16_gemm_residual_gb300", "csrc")
    for name in sorted(KERNEL_SOURCES.get(kernel, ())):
        try:
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
        except OSError:
            h.update(name.encode() + b"\0missing")
    return h.hexdigest()[:16]


def committed_traffic(kernel: str):
    """dram bytes per launch from the committed ncu summary for `kernel`, if it
    was taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_traffic.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_digest") != kernel_source_digest(kernel):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ stats
def summarize(samples):
    """Median, p10, p90 (linear interpolation), mean and cv% of samples (the
    vLLM benchmark page's summary statistics)."""
    ordered = sorted(samples)

    def pct(f):
        pos = f * (len(ordered) - 1)
        lo, hi = math.floor(pos), math.ceil(pos)
        if lo == hi:
            return ordered[lo]
        w = pos - lo
        return ordered[lo] * (1 - w) + ordered[hi] * w

    mean = statistics.mean(samples)
    return {"median_us": statistics.median(samples), "p10_us": pct(0.1), "p90_us": pct(0.9),
            "mean_us": mean, "cv_pct": statistics.pstdev(samples) / mean * 100.0 if mean else 0.0}


# ------------------------------------------------------------------ dist
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_max(value: float, ws: int, device=None) -> float:
    """Max of a host float over ranks (timing aggregation; no data-path collective)."""
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_step: float, ws: int, steps: int, slowest_ms: float) -> float:
    """Whole-job throughput: the bytes every rank processed (each rank runs the
    same step on its own GPU: replicas) over the slowest rank's time."""
    return bytes_per_step * ws * steps / (slowest_ms * 1e-3) / 1e9


def dist_barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist

        dist.barrier()


# ------------------------------------------------------------------ workload
def make_workload(device, m_list=M_LIST, copies=COPIES):
    """Rotating W copies (seed s) shared by every M; per-M activation and
    per-(M, copy) residuals.  Generated on the host, copied to the device."""
    import torch

    from skinny_bf16_gemm_residual_gb300 import inputs

    Ws_cpu = [inputs.make_weights(N_DIM, K_DIM, seed=s) for s in range(copies)]
    Ws = [w.to(device) for w in Ws_cpu]
    per_m = {}
    for M in m_list:
        A_cpu = inputs.make_rows(M, K_DIM, seed=10_000 + M)
        Rs_cpu = [inputs.make_rows(M, N_DIM, seed=20_000 + 100 * M + s) for s in range(copies)]
        per_m[M] = {
            "A_cpu": A_cpu, "R_cpu": Rs_cpu,
            "A": A_cpu.to(device), "R": [r.to(device) for r in Rs_cpu],
            "Y": [torch.empty((M, N_DIM), dtype=torch.bfloat16, device=device) for _ in range(copies)],
        }
    return Ws_cpu, Ws, per_m


def capture(calls, stream):
    """Eager warm-up of every call, then one CUDA graph holding all of them."""
    import torch

    with torch.cuda.stream(stream):
        for fn in calls:
            fn()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for fn in calls:
            fn()
    return g


def time_graph(g, stream, replays: int, repeats: int):
    import torch

    out = []
    with torch.cuda.stream(stream):  # replay() launches on the current stream
        for _ in range(repeats):
            s = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            s.record(stream)
            for _ in range(replays):
                g.replay()
            e.record(stream)
            e.synchronize()
            out.append(s.elapsed_time(e) * 1000.0 / replays)  # us per replay
    return out


def time_calls(calls, stream, replays: int, repeats: int, warm: int = 20) -> dict:
    """One CUDA graph of `calls` (eager warm-up first), `warm` untimed replays,
    then `repeats` x `replays` between CUDA events; summary per call."""
    import torch

    g = capture(calls, stream)
    with torch.cuda.stream(stream):
        for _ in range(warm):
            g.replay()
    stream.synchronize()
    s = summarize([t / len(calls) for t in time_graph(g, stream, replays, repeats)])
    del g
    return s


def call_metrics(M: int, s: dict, peaks: dict) -> dict:
    """Per-call figures of one timing summary: GB/s and TFLOP/s of the
    algorithmic bytes and FLOPs, their fractions of the measured peaks (the
    burst tensor peak for a kernel timed on its own, the sustained one beside
    it), and the fraction of the roofline time max(bytes / HBM peak,
    FLOPs / tensor peak)."""
    us = s["median_us"]
    gbs = alg_bytes(M) / (us * 1e-6) / 1e9
    tflops = alg_flops(M) / (us * 1e-6) / 1e12
    roof_us = max(alg_bytes(M) / (peaks["hbm_gbs"] * 1e9), alg_flops(M) / (peaks["bf16_tflops"] * 1e12)) * 1e6
    return {"us_per_call": us, "p10_us": s["p10_us"], "p90_us": s["p90_us"], "cv_pct": s["cv_pct"],
            "gbs": gbs, "frac_of_hbm_peak": gbs / peaks["hbm_gbs"],
            "tflops": tflops, "frac_of_tensor_peak": tflops / peaks["bf16_tflops"],
            "frac_of_tensor_peak_sustained": tflops / peaks["bf16_tflops_sustained"],
            "roofline_us": roof_us, "frac_of_roofline": roof_us / us,
            "bound": "tensor" if tensor_bound(M, peaks) else "hbm"}


def addmm_calls(A, Ws, Rs, Ys, stream):
    """The cuBLAS comparator of the vLLM benchmark page (its `addmm` backend):
    Y = R + A . W^T by torch.addmm into the output buffer, one call per copy."""
    import torch

    def one(c):
        def f():
            with torch.cuda.stream(stream):
                torch.addmm(Rs[c], A, Ws[c].t(), out=Ys[c])
        return f
    return [one(c) for c in range(len(Ws))]


def run_sweep(sgr, Ws, device, stream, peaks: dict, m_list, paths, replays: int, repeats: int) -> dict:
    """Every kernel path in `paths` (plus the library's automatic choice and
    cuBLAS addmm) at each M, each as one CUDA graph of one call per rotating W
    copy, PDL on.  A path that cannot run the shape is recorded as such."""
    import torch

    from skinny_bf16_gemm_residual_gb300 import inputs

    out = {}
    for M in m_list:
        A = inputs.make_rows(M, K_DIM, seed=10_000 + M).to(device)
        Rs = [inputs.make_rows(M, N_DIM, seed=20_000 + 100 * M + c).to(device) for c in range(COPIES)]
        Ys = [torch.empty((M, N_DIM), dtype=torch.bfloat16, device=device) for _ in range(COPIES)]
        auto = PATH_NAMES.get(sgr.sgr_select_path(M, N_DIM, K_DIM), "?")
        entry = {"library_choice": auto, "paths": {}}
        for name in list(paths) + ["auto"]:
            cfg = None if name == "auto" else sgr.make_config(path=PATH_IDS[name])
            calls = [lambda c=c, cfg=cfg: sgr.skinny_gemm_residual_ex(A, Ws[c], Rs[c], Ys[c], config=cfg,
                                                                      stream=stream) for c in range(COPIES)]
            try:
                calls[0]()
                stream.synchronize()
            except sgr.SgrError as e:
                entry["paths"][name] = {"unsupported": str(e)}
                continue
            entry["paths"][name] = call_metrics(M, time_calls(calls, stream, replays, repeats), peaks)
        entry["paths"]["cublas_addmm"] = call_metrics(
            M, time_calls(addmm_calls(A, Ws, Rs, Ys, stream), stream, replays, repeats), peaks)
        out[str(M)] = entry
        del A, Rs, Ys
    return out


# ------------------------------------------------------------------ CPU arms
ARM_CORES = {("0x41", "0xd4f"): "Arm Neoverse V2", ("0x41", "0xd40"): "Arm Neoverse V1",
             ("0x41", "0xd49"): "Arm Neoverse N2", ("0x41", "0xd0c"): "Arm Neoverse N1"}


def cpu_model(cpuinfo: str | None = None) -> str:
    """The host CPU's name as /proc/cpuinfo gives it (x86 "model name"; on Arm,
    which lists no name, the core named from its implementer and part codes)."""
    if cpuinfo is None:
        try:
            with open("/proc/cpuinfo") as f:
                cpuinfo = f.read()
        except OSError:
            cpuinfo = ""
    fields = {}
    for line in cpuinfo.splitlines():
        if ":" in line:
            k, v = line.split(":", 1)
            fields.setdefault(k.strip(), v.strip())
    for key in ("model name", "Model", "Hardware"):
        if fields.get(key):
            return fields[key]
    if "CPU part" in fields:
        impl, part = fields.get("CPU implementer", "?"), fields["CPU part"]
        name = ARM_CORES.get((impl, part))
        return f"{name} (implementer {impl}, part {part})" if name else f"{platform.machine()} implementer {impl} part {part}"
    return platform.machine() or "unknown"


def cpu_oracle_rate(Ws_cpu, per_m_cpu, m_list, budget_s: float, n_rows: int | None = None,
                    threads: int | None = None):
    """Time the oracle on the workload, bounded by budget_s, on `threads` host
    threads (default: all cores).  The threads split the output rows, so the
    bits do not depend on the count.
    Returns (GB/s of algorithmic bytes, threads, sample description, seconds)."""
    import oracle

    threads = threads or os.cpu_count() or 1
    lib = oracle.load()
    n_rows = n_rows or N_DIM
    done_bytes, t0, calls = 0, time.perf_counter(), 0
    while True:
        for M in m_list:
            A = per_m_cpu[M]["A_cpu"]
            R = per_m_cpu[M]["R_cpu"][calls % len(Ws_cpu)][:, :n_rows]
            W = Ws_cpu[calls % len(Ws_cpu)][:n_rows]
            lib.gemm_residual(A, W, R, threads=threads)
            done_bytes += alg_bytes(M, n_rows, K_DIM)
        calls += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    desc = (f"{calls} pass(es) over M in {list(m_list)} with the first {n_rows} of {N_DIM} "
            f"output columns (K={K_DIM}), FP64 C oracle, {threads} threads")
    return done_bytes / el / 1e9, threads, desc, el


def run_reference(args):
    """Reference arm: the CPU oracle as it stands, on the host cores."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    from skinny_bf16_gemm_residual_gb300 import inputs

    m_list = tuple(int(x) for x in args.m_list.split(","))
    Ws_cpu = [inputs.make_weights(N_DIM, K_DIM, seed=s) for s in range(COPIES)]
    per_m = {M: {"A_cpu": inputs.make_rows(M, K_DIM, seed=10_000 + M),
                 "R_cpu": [inputs.make_rows(M, N_DIM, seed=20_000 + 100 * M + s) for s in range(COPIES)]}
             for M in m_list}
    import oracle

    lib = oracle.load()
    threads = os.cpu_count() or 1
    # Size one step so that warmup + steps fit in about args.ref_budget seconds.
    t0 = time.perf_counter()
    probe_rows = 256
    for M in m_list:
        lib.gemm_residual(per_m[M]["A_cpu"], Ws_cpu[0][:probe_rows], per_m[M]["R_cpu"][0][:, :probe_rows],
                          threads=threads)
    per_row = (time.perf_counter() - t0) / probe_rows
    total_steps = args.steps + args.warmup
    rows = int(args.ref_budget / max(total_steps, 1) / max(per_row, 1e-9))
    rows = max(8, min(N_DIM, rows // 8 * 8))
    times, nbytes = [], sum(alg_bytes(M, rows, K_DIM) for M in m_list)
    for i in range(total_steps):
        c = i % COPIES
        t0 = time.perf_counter()
        for M in m_list:
            lib.gemm_residual(per_m[M]["A_cpu"], Ws_cpu[c][:rows], per_m[M]["R_cpu"][c][:, :rows],
                              threads=threads)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    total = sum(times)
    value = nbytes * len(times) / total / 1e9
    sample = (f"each step: one call per M in {list(m_list)} on the first {rows} of {N_DIM} output "
              f"columns (W rows), K={K_DIM}, rotating 4 W copies; FP64 C oracle")
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "impl": "reference",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / len(times) * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name(m_list), "sample_columns": rows,
                   "parallelism": "host cores, rank 0 only"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample,
                         "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm
def run_ours(args):
    import torch

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    device = torch.device("cuda", torch.cuda.current_device())
    import skinny_bf16_gemm_residual_gb300 as sgr

    sgr.sgr_init(device.index)
    m_list = tuple(int(x) for x in args.m_list.split(","))
    Ws_cpu, Ws, per_m = make_workload(device, m_list)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    w_total = COPIES * N_DIM * K_DIM * 2
    assert w_total > 1.5 * l2, "rotating W copies must exceed L2"
    stream = torch.cuda.Stream(device=device)

    def call(M, c):
        d = per_m[M]
        return lambda: sgr.skinny_gemm_residual(d["A"], Ws[c], d["R"][c], d["Y"][c], stream=stream)

    step_calls = [call(M, c) for M in m_list for c in range(COPIES)]
    launches_per_step = len(step_calls)
    bytes_per_step = sum(alg_bytes(M) for M in m_list for _ in range(COPIES))
    g_step = capture(step_calls, stream)

    # per-M microseconds per call: one graph of the 4 copies, repeats x replays;
    # the cuBLAS addmm comparator the same way; the first M measured again
    # after the others (a measurement-order check)
    per_m_out = {}
    peaks, peak_src = load_peaks()
    for M in (() if args.skip_per_m else m_list):
        s = time_calls([call(M, c) for c in range(COPIES)], stream, args.replays, args.repeats)
        per_m_out[str(M)] = {**call_metrics(M, s, peaks),
                             "path": PATH_NAMES.get(sgr.sgr_select_path(M, N_DIM, K_DIM), "?")}
        if not args.skip_cublas:
            d = per_m[M]
            sc = time_calls(addmm_calls(d["A"], Ws, d["R"], d["Y"], stream), stream, args.replays, args.repeats)
            per_m_out[str(M)]["cublas_addmm"] = call_metrics(M, sc, peaks)
    if per_m_out and len(m_list) > 1:
        M = m_list[0]
        s = time_calls([call(M, c) for c in range(COPIES)], stream, args.replays, args.repeats)
        per_m_out[str(M)]["measured_again_last"] = call_metrics(M, s, peaks)

    # headline: K timed steps of the whole M sweep, the K-step region repeated
    # (each repeat bracketed by a barrier and a device synchronise, timed with
    # CUDA events on the launch stream) until the repeats span about
    # args.headline_seconds, so that the clock sampler sees the load
    clocks = ClockSampler(device.index)
    clocks.start()
    with torch.cuda.stream(stream):  # replay() launches on the current stream
        for _ in range(args.warmup):
            g_step.replay()
    stream.synchronize()

    def timed_region():
        dist_barrier(ws)
        torch.cuda.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(args.steps):
                g_step.replay()
            ev1.record(stream)
        ev1.synchronize()
        torch.cuda.synchronize()
        dist_barrier(ws)
        return ev0.elapsed_time(ev1)

    first_ms = timed_region()
    repeats = max(args.min_headline_repeats, math.ceil(args.headline_seconds * 1e3 / max(first_ms, 1e-3)))
    repeats = int(dist_max(float(repeats), ws, device))  # every rank runs the same count
    region_ms = [first_ms] + [timed_region() for _ in range(repeats - 1)]
    clk = clocks.stop()
    if ws > 1:
        t = torch.tensor(region_ms, dtype=torch.float64, device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        region_ms = t.tolist()  # per repeat, the slowest rank
    rs = summarize(region_ms)  # milliseconds here, despite the key names
    elapsed_ms = rs["median_us"]
    ms_per_step = elapsed_ms / args.steps
    value = job_gbs(bytes_per_step, ws, args.steps, elapsed_ms)
    headline = {"repeats": repeats, "steps_per_repeat": args.steps,
                "ms_per_repeat": {"median": rs["median_us"], "p10": rs["p10_us"], "p90": rs["p90_us"],
                                  "cv_pct": rs["cv_pct"]},
                "gbs_p10_time": job_gbs(bytes_per_step, ws, args.steps, rs["p10_us"]),
                "gbs_p90_time": job_gbs(bytes_per_step, ws, args.steps, rs["p90_us"]),
                "seconds_timed": sum(region_ms) / 1e3,
                "note": "value and ms_per_step from the median repeat of the K-step region"}

    # end to end through the public call with host buffers (pinned), W resident
    e2e_out = None
    if not args.skip_e2e:
        e2e = run_e2e(sgr, per_m, Ws, m_list, device, stream, max(3, min(args.steps, args.e2e_steps)))
        e2e_seconds = dist_max(e2e["seconds"], ws, device)  # slowest rank
        e2e_out = {"value": bytes_per_step * ws * e2e["steps"] / e2e_seconds / 1e9, "unit": "GB/s",
                   "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                   "steps": e2e["steps"],
                   "note": "host wall clock; every step copies its inputs in and its outputs out (pinned); "
                           "steps pipelined over two buffer sets and separate copy streams"}

    transition = None if (args.skip_sweeps or rank != 0) else run_sweep(
        sgr, Ws, device, stream, peaks, TRANSITION_M, ("rows", "tc", "tile", "pair"), args.sweep_replays, args.repeats)
    compute_bound = None if (args.skip_sweeps or rank != 0) else run_sweep(
        sgr, Ws, device, stream, peaks, COMPUTE_M, ("tile", "pair"), args.sweep_replays, args.repeats)
    chain = None if (args.skip_chain or rank != 0) else run_chain(sgr, device, stream)
    grouped = None if (args.skip_grouped or rank != 0) else run_grouped(sgr, device, stream)
    w8 = None if (args.skip_w8 or rank != 0) else run_w8(sgr, device, stream, peaks)
    w4 = None if (args.skip_w4 or rank != 0) else run_w4(sgr, device, stream, peaks)
    down = None if (args.skip_down or rank != 0 or (N_DIM, K_DIM) != (7168, 3584)) else run_down(
        sgr, device, stream, peaks)

    if rank != 0:
        return 0

    avg_launch_s = elapsed_ms * 1e-3 / (args.steps * launches_per_step)  # median repeat
    achieved = bytes_per_step / launches_per_step / avg_launch_s / 1e9
    # dominant kernel: the path with the largest share of the step's time
    share = {}
    for M in m_list:
        path = PATH_NAMES.get(sgr.sgr_select_path(M, N_DIM, K_DIM), "?")
        us = per_m_out[str(M)]["us_per_call"] if str(M) in per_m_out else 1.0
        share[path] = share.get(path, 0.0) + us
    dominant_path = max(share, key=share.get)
    dominant = KERNEL_NAMES.get(dominant_path, dominant_path)
    traffic = committed_traffic(dominant)
    flops_per_step = sum(alg_flops(M) for M in m_list) * COPIES
    if all(tensor_bound(M, peaks) for M in m_list):
        t_ach = flops_per_step / launches_per_step / avg_launch_s / 1e12
        roofline_bound = {"bound": "tensor", "achieved": t_ach, "peak": peaks["bf16_tflops"],
                          "unit": "TFLOP/s", "frac": t_ach / peaks["bf16_tflops"]}
    else:
        roofline_bound = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                          "frac": achieved / peaks["hbm_gbs"]}
    roofline = {
        **roofline_bound, "traffic": traffic, "peak_source": peak_src,
        "kernel": dominant,
        "kernels_in_step": {KERNEL_NAMES.get(k, k): round(v / sum(share.values()), 3) for k, v in share.items()},
        "bytes_per_launch": bytes_per_step / launches_per_step,
        "flops_per_launch": flops_per_step / launches_per_step,
        "note": "algorithmic bytes 2*(N*K + M*K + 2*M*N) (or FLOPs 2*M*N*K when every M of the step "
                "is past the ridge point) per call averaged over the step's calls / average launch "
                "duration over the timed region (CUDA events on the launch stream)",
    }
    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        rate, threads, desc, secs = cpu_oracle_rate(Ws_cpu, per_m, m_list, args.cpu_budget)
        rate1, _, desc1, secs1 = cpu_oracle_rate(Ws_cpu, per_m, m_list, args.cpu_single_budget, threads=1)
        cpu = {"value": rate, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": desc,
               "seconds": secs, "cpu_model": cpu_model(),
               "single_thread": {"value": rate1, "unit": "GB/s", "sample": desc1, "seconds": secs1}}
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {
            "workload": workload_name(m_list),
            "calls_per_step": launches_per_step, "l2": "inputs larger than L2 (4 W copies = "
            f"{w_total / 1e6:.0f} MB vs L2 {l2 / 1e6:.0f} MB); no flush",
            "launch": "one CUDA graph per step, PDL on", "parallelism": "replicas" if ws > 1 else "single GPU",
        },
        "headline": headline,
        "per_m": per_m_out,
        "transition": transition,
        "compute_bound": compute_bound,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e_out,
        "chain": chain,
        "grouped": grouped,
        "w8": w8,
        "w4": w4,
        "down_projection": down,
        "gpu_launches": repeats * args.steps * launches_per_step,
        "clocks": clk,
        "peaks": {"hbm_gbs": peaks["hbm_gbs"], "bf16_tflops": peaks["bf16_tflops"],
                  "bf16_tflops_sustained": peaks["bf16_tflops_sustained"], "source": peak_src},
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def run_chain(sgr, device, stream, layers: int = 8, M: int = 4, replays: int = 50, repeats: int = 9):
    """The chain of dependent projections: layer i reads A_i = Y_{i-1}[:, :K]
    (row stride N) and its own W_i (8 distinct weights, 411 MB, so none is in
    L2) and R_i; one CUDA graph of all layers, timed with programmatic
    dependent launch on and off.  Returns us per layer for both."""
    import torch

    from skinny_bf16_gemm_residual_gb300 import inputs

    Ws = [inputs.make_weights(N_DIM, K_DIM, seed=1000 + i).to(device) for i in range(layers)]
    Rs = [inputs.make_rows(M, N_DIM, seed=2000 + i).to(device) for i in range(layers)]
    A0 = inputs.make_rows(M, K_DIM, seed=3000).to(device)
    Ys = [torch.empty((M, N_DIM), dtype=torch.bfloat16, device=device) for _ in range(layers)]
    out = {}
    for name, flags in (("pdl", 0), ("no_pdl", sgr.SGR_FLAG_NO_PDL)):
        def layer(i, flags=flags):
            A = A0 if i == 0 else Ys[i - 1][:, :K_DIM]
            return lambda: sgr.skinny_gemm_residual_ex(A, Ws[i], Rs[i], Ys[i], flags=flags, stream=stream)

        g = capture([layer(i) for i in range(layers)], stream)
        with torch.cuda.stream(stream):
            for _ in range(5):
                g.replay()
        stream.synchronize()
        samples = [t / layers for t in time_graph(g, stream, replays, repeats)]
        out[name] = summarize(samples)["median_us"]
        del g
    gbs = alg_bytes(M) / (out["pdl"] * 1e-6) / 1e9
    return {"layers": layers, "m": M, "us_per_layer": out["pdl"], "us_per_layer_no_pdl": out["no_pdl"],
            "pdl_saving_us": out["no_pdl"] - out["pdl"], "gbs": gbs,
            "note": "graph of 8 dependent calls, A_i = Y_{i-1}[:, :K] (lda = N), distinct W_i"}


def run_grouped(sgr, device, stream, experts: int = 8, tokens: int = 16, top_k: int = 2,
                replays: int = 50, repeats: int = 9):
    """Mixture-of-experts step: `tokens` tokens routed top-k over `experts`
    experts (seeded synthetic routing), each expert its own W_e; one grouped
    launch versus one call per expert, both in a CUDA graph with PDL."""
    import numpy as np
    import torch

    from skinny_bf16_gemm_residual_gb300 import inputs

    rng = np.random.default_rng(2024)
    choice = np.stack([rng.choice(experts, size=top_k, replace=False) for _ in range(tokens)])
    counts = np.bincount(choice.ravel(), minlength=experts).tolist()
    Ws = [inputs.make_weights(N_DIM, K_DIM, seed=4000 + e).to(device) for e in range(experts)]
    As = [inputs.make_rows(m, K_DIM, seed=5000 + e).to(device) for e, m in enumerate(counts)]
    Rs = [inputs.make_rows(m, N_DIM, seed=6000 + e).to(device) for e, m in enumerate(counts)]
    Ys = [torch.empty((m, N_DIM), dtype=torch.bfloat16, device=device) for m in counts]
    problems = list(zip(As, Ws, Rs, Ys))
    active = [(A, W, R, Y) for A, W, R, Y in problems if A.shape[0] > 0]
    nbytes = sum(alg_bytes(A.shape[0]) for A, _, _, _ in active)
    out = {}
    for name, calls in (
            ("grouped", [lambda: sgr.skinny_gemm_residual_grouped(problems, stream=stream)]),
            ("per_expert", [lambda A=A, W=W, R=R, Y=Y: sgr.skinny_gemm_residual(A, W, R, Y, stream=stream)
                            for A, W, R, Y in active])):
        g = capture(calls, stream)
        with torch.cuda.stream(stream):
            for _ in range(5):
                g.replay()
        stream.synchronize()
        out[name] = summarize(time_graph(g, stream, replays, repeats))["median_us"]
        del g
    return {"experts": experts, "tokens": tokens, "top_k": top_k, "tokens_per_expert": counts,
            "us_grouped": out["grouped"], "us_per_expert_calls": out["per_expert"],
            "gbs_grouped": nbytes / (out["grouped"] * 1e-6) / 1e9,
            "gbs_per_expert_calls": nbytes / (out["per_expert"] * 1e-6) / 1e9,
            "note": "one step = all experts with tokens; bytes = sum over those experts of 2*(N*K + M*K + 2*M*N)"}


def run_w8(sgr, device, stream, peaks: dict, m_list=(1, 2, 4, 16), copies: int = 8, replays: int = 50,
           repeats: int = 9):
    """Low-bit weight leg: the same projection with FP8 E4M3 weights and a
    per-column scale (skinny_gemm_residual_w8).  Per M, one CUDA graph of
    `copies` calls over distinct weight copies (8 x 25.7 MB, more than L2),
    PDL on.  Bytes per call = N*K (codes) + 4N (scales) + 2MK + 4MN."""
    import torch

    from skinny_bf16_gemm_residual_gb300 import inputs

    qs = [inputs.make_problem_w8(1, N_DIM, K_DIM, seed=7000 + c) for c in range(copies)]
    Wq = [q.Wq.to(device) for q in qs]
    Sc = [q.scale.to(device) for q in qs]
    rows = []
    for M in m_list:
        A = inputs.make_rows(M, K_DIM, seed=8000 + M).to(device)
        R = inputs.make_rows(M, N_DIM, seed=9000 + M).to(device)
        Y = torch.empty((M, N_DIM), dtype=torch.bfloat16, device=device)
        calls = [lambda c=c: sgr.skinny_gemm_residual_w8(A, Wq[c], Sc[c], R, Y, stream=stream) for c in range(copies)]
        g = capture(calls, stream)
        with torch.cuda.stream(stream):
            for _ in range(5):
                g.replay()
        stream.synchronize()
        us = summarize([t / copies for t in time_graph(g, stream, replays, repeats)])["median_us"]
        del g
        nbytes = N_DIM * K_DIM + 4 * N_DIM + 2 * M * K_DIM + 4 * M * N_DIM
        gbs = nbytes / (us * 1e-6) / 1e9
        rows.append({"m": M, "kernel": "w8s_kernel" if M <= 8 else "w8_rows_kernel",
                     "us": us, "bytes": nbytes, "gbs": gbs,
                     "frac_of_hbm_peak": gbs / peaks["hbm_gbs"] if peaks.get("hbm_gbs") else None})
    return {"per_m": rows,
            "note": "FP8 E4M3 weights + FP32 per-column scale, BF16 A/R/Y; graph of 8 calls over distinct weight "
                    "copies; the library's own kernel choice (FP8 tensor-core kernel with split activations for "
                    "M <= 8, the widening row-slab kernel above)"}


def run_down(sgr, device, stream, peaks: dict, m_list=(1, 4, 16, 32, 64), replays: int = 50, repeats: int = 9):
    """The block's other projection, K = 7168 -> N = 3584 (the down-projection),
    when the headline runs the up-projection: per M, the library's own choice
    (the row slab with the 2-CTA K split up to 64 tokens) and cuBLAS `addmm`,
    each as one CUDA graph of COPIES calls over distinct weight copies (4 x
    51 MB, more than L2), PDL on."""
    import torch

    from skinny_bf16_gemm_residual_gb300 import inputs

    N, K = K_DIM, N_DIM
    Ws = [inputs.make_weights(N, K, seed=11_000 + c).to(device) for c in range(COPIES)]
    rows = []
    for M in m_list:
        A = inputs.make_rows(M, K, seed=12_000 + M).to(device)
        Rs = [inputs.make_rows(M, N, seed=13_000 + 100 * M + c).to(device) for c in range(COPIES)]
        Ys = [torch.empty((M, N), dtype=torch.bfloat16, device=device) for _ in range(COPIES)]
        ours = time_calls([lambda c=c: sgr.skinny_gemm_residual(A, Ws[c], Rs[c], Ys[c], stream=stream)
                           for c in range(COPIES)], stream, replays, repeats)
        ref = time_calls(addmm_calls(A, Ws, Rs, Ys, stream), stream, replays, repeats)
        gbs = alg_bytes(M, N, K) / (ours["median_us"] * 1e-6) / 1e9
        rows.append({"m": M, "path": PATH_NAMES.get(sgr.sgr_select_path(M, N, K), "?"),
                     "us": ours["median_us"], "p10_us": ours["p10_us"], "p90_us": ours["p90_us"],
                     "gbs": gbs, "frac_of_hbm_peak": gbs / peaks["hbm_gbs"],
                     "cublas_addmm_us": ref["median_us"]})
    del Ws
    return {"n": N, "k": K, "per_m": rows,
            "note": "down-projection of the same block; graph of 4 calls over distinct weight copies; "
                    "the library's choice and cuBLAS addmm under the same protocol"}


def run_w4(sgr, device, stream, peaks: dict, m_list=(1, 2, 4, 16), copies: int = 8, replays: int = 50,
           repeats: int = 9):
    """NVFP4 weight leg: the same projection with E2M1 codes, one E4M3 scale
    per 16 elements and an FP32 tensor scale (skinny_gemm_residual_w4).  Per
    M, one CUDA graph of `copies` calls over distinct weight copies (8 x 14.5
    MB, more than L2), PDL on.  Bytes per call = N*K/2 (codes) + N*K/16
    (block scales) + 2MK + 4MN."""
    import torch

    from skinny_bf16_gemm_residual_gb300 import inputs

    qs = [inputs.make_problem_w4(1, N_DIM, K_DIM, seed=7100 + c) for c in range(copies)]
    Wq4 = [q.Wq4.to(device) for q in qs]
    Bs = [q.bs.to(device) for q in qs]
    rows = []
    for M in m_list:
        A = inputs.make_rows(M, K_DIM, seed=8100 + M).to(device)
        R = inputs.make_rows(M, N_DIM, seed=9100 + M).to(device)
        Y = torch.empty((M, N_DIM), dtype=torch.bfloat16, device=device)
        calls = [lambda c=c: sgr.skinny_gemm_residual_w4(A, Wq4[c], Bs[c], qs[c].gs, R, Y, stream=stream)
                 for c in range(copies)]
        g = capture(calls, stream)
        with torch.cuda.stream(stream):
            for _ in range(5):
                g.replay()
        stream.synchronize()
        us = summarize([t / copies for t in time_graph(g, stream, replays, repeats)])["median_us"]
        del g
        passes = (M + 3) // 4 if M <= 1 else (M + 127) // 128  # CUDA-core kernel: 4 tokens per pass
        wbytes = N_DIM * K_DIM // 2 + N_DIM * K_DIM // 16
        nbytes = wbytes + 2 * M * K_DIM + 4 * M * N_DIM
        gbs = nbytes / (us * 1e-6) / 1e9
        rows.append({"m": M, "kernel": "simt_skinny_kernel<nvfp4>" if M <= 1 else "w8_rows_kernel<nvfp4>",
                     "passes": passes, "us": us, "bytes": nbytes,
                     "bytes_streamed": passes * wbytes + 2 * M * K_DIM + 4 * M * N_DIM, "gbs": gbs,
                     "frac_of_hbm_peak": gbs / peaks["hbm_gbs"] if peaks.get("hbm_gbs") else None})
    return {"per_m": rows,
            "note": "NVFP4 weights (E2M1 codes, E4M3 scale per 16 elements, FP32 tensor scale), BF16 A/R/Y; graph "
                    "of 8 calls over distinct weight copies; the library's choice: CUDA-core kernel for M = 1, "
                    "tensor-core widening kernel above; gbs counts each weight byte once"}


def run_e2e(sgr, per_m, Ws, m_list, device, stream, steps: int):
    """Each step: one host->device copy of the step's inputs (A for every M,
    R for every call) from a pinned host buffer, the public call for every
    (M, copy), and one device->host copy of every Y into pinned host memory;
    W stays resident (weights).  Steps are pipelined over two buffer sets:
    the input copy runs on its own stream, the calls on `stream`, the output
    copy on a third stream, ordered by events, and before a buffer set is
    reused the host waits until that set's results have arrived.  Every
    step's copies are inside the timed region, which ends when the last
    step's results are in host memory."""
    import torch

    # one contiguous pinned staging buffer per direction, with views per operand
    in_sizes, out_sizes = [], []
    for M in m_list:
        in_sizes.append(M * K_DIM)
        in_sizes += [M * N_DIM] * COPIES
        out_sizes += [M * N_DIM] * COPIES
    h_in = torch.empty(sum(in_sizes), dtype=torch.bfloat16).pin_memory()
    pos_in = 0
    layout = []  # (a offset, r offset, y offset, M, copy) in elements
    pos_out = 0
    for M in m_list:
        d = per_m[M]
        a_off = pos_in
        h_in[pos_in:pos_in + M * K_DIM].copy_(d["A_cpu"].reshape(-1))
        pos_in += M * K_DIM
        for c in range(COPIES):
            h_in[pos_in:pos_in + M * N_DIM].copy_(d["R_cpu"][c].reshape(-1))
            layout.append((a_off, pos_in, pos_out, M, c))
            pos_in += M * N_DIM
            pos_out += M * N_DIM
    sets = []
    for _ in range(2):
        d_in = torch.empty(sum(in_sizes), dtype=torch.bfloat16, device=device)
        d_out = torch.empty(sum(out_sizes), dtype=torch.bfloat16, device=device)
        h_out = torch.empty(sum(out_sizes), dtype=torch.bfloat16).pin_memory()
        calls = [(d_in.data_ptr() + 2 * a, Ws[c].data_ptr(), d_in.data_ptr() + 2 * r, d_out.data_ptr() + 2 * y, M)
                 for a, r, y, M, c in layout]
        sets.append({"d_in": d_in, "d_out": d_out, "h_out": h_out, "calls": calls,
                     "ev_in": torch.cuda.Event(), "ev_out": torch.cuda.Event(), "ev_host": torch.cuda.Event(),
                     "used": False})
    h2d = h_in.numel() * 2
    d2h = sets[0]["h_out"].numel() * 2
    s = stream.cuda_stream
    s_in, s_out = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)

    def launch_step(i):
        st = sets[i % 2]
        if st["used"]:
            st["ev_host"].synchronize()  # that set's previous results are in host memory
        st["used"] = True
        with torch.cuda.stream(s_in):
            st["d_in"].copy_(h_in, non_blocking=True)
            st["ev_in"].record(s_in)
        stream.wait_event(st["ev_in"])
        for A, W, R, Y, M in st["calls"]:
            rc = sgr.skinny_gemm_residual_ptr(A, W, R, Y, M, N_DIM, K_DIM, s)
            if rc != sgr.SGR_OK:
                raise sgr.SgrError(rc, "skinny_gemm_residual")
        st["ev_out"].record(stream)
        s_out.wait_event(st["ev_out"])
        with torch.cuda.stream(s_out):
            st["h_out"].copy_(st["d_out"], non_blocking=True)
            st["ev_host"].record(s_out)

    def finish():
        for st in sets:
            if st["used"]:
                st["ev_host"].synchronize()

    for i in range(3):
        launch_step(i)
    finish()
    t0 = time.perf_counter()
    for i in range(steps):
        launch_step(i)
    finish()
    secs = time.perf_counter() - t0
    return {"seconds": secs, "steps": steps, "h2d": h2d, "d2h": d2h}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--m-list", default=",".join(str(m) for m in M_LIST))
    ap.add_argument("--repeats", type=int, default=21)
    ap.add_argument("--replays", type=int, default=200)
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--cpu-single-budget", type=float, default=4.0,
                    help="seconds of single-threaded oracle time (cpu_baseline.single_thread)")
    ap.add_argument("--ref-budget", type=float, default=90.0, help="seconds for the reference arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--skip-per-m", action="store_true", help="skip the per-M repeat/replay timing")
    ap.add_argument("--skip-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--skip-chain", action="store_true", help="skip the 8-layer dependent chain leg")
    ap.add_argument("--skip-grouped", action="store_true", help="skip the mixture-of-experts grouped leg")
    ap.add_argument("--skip-w8", action="store_true", help="skip the FP8-weight leg")
    ap.add_argument("--skip-w4", action="store_true", help="skip the NVFP4-weight leg")
    ap.add_argument("--skip-down", action="store_true", help="skip the down-projection (N 3584, K 7168) leg")
    ap.add_argument("--skip-sweeps", action="store_true",
                    help="skip the transition (M = 32-128) and compute-bound (M = 256-1024) legs")
    ap.add_argument("--skip-cublas", action="store_true", help="skip the cuBLAS addmm rows of the per-M leg")
    ap.add_argument("--sweep-replays", type=int, default=100, help="replays per repeat in the M = 32-1024 legs")
    ap.add_argument("--headline-seconds", type=float, default=2.0,
                    help="repeat the K-step timed region until the repeats span about this long")
    ap.add_argument("--min-headline-repeats", type=int, default=5)
    ap.add_argument("--n", type=int, default=7168, help="output features (the headline shape is 7168)")
    ap.add_argument("--k", type=int, default=3584, help="input features (the headline shape is 3584)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    set_shape(args.n, args.k)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
