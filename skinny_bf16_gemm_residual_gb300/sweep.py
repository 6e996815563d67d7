"""Configuration sweep for the skinny GEMM + residual kernels (GPU).

The analogue of the sweep mode of the vLLM "benchmark_k3_cutedsl_residual.py"
page: for each M, every candidate launch configuration of each kernel path is
timed by batched CUDA-graph replay over rotating weight/residual copies that
together exceed L2, and one JSON row per (M, path, config) is written.  A
`torch.addmm` (cuBLAS) row under the same protocol is included as context.
The per-M table compiled into the library is generated from these rows by
``gen_table.py``.  The paths ``w8`` (widening tensor-core FP8-weight kernel), ``w8s`` (FP8
tensor-core kernel with split activations) and
``w8simt`` (CUDA-core FP8-weight kernel) time ``skinny_gemm_residual_w8`` over
rotating copies of per-column-quantised E4M3 weights; ``w4`` (tensor-core
widening kernel) and ``w4simt`` (CUDA-core kernel) time
``skinny_gemm_residual_w4`` over rotating copies of NVFP4-quantised weights.
Their rows are for choosing those entry points' defaults and are not part of
the BF16 table.

    python -m skinny_bf16_gemm_residual_gb300.sweep --m 1 2 4 8 16 --output sweep.jsonl
    python -m skinny_bf16_gemm_residual_gb300.sweep --paths w8,w8simt --copies 8 --output sweep_w8.jsonl

Rows are written as soon as they are timed.  With ``--resume`` the output file
is appended to and every (M, N, K, backend, configuration) already in it is
skipped, so an interrupted sweep continues where it stopped.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import sys

import torch

from . import binding as sgr
from . import inputs


def candidate_configs_w8s(M: int, grid: str) -> list[dict]:
    """Launch configurations of the FP8 tensor-core kernel with split
    activations (M <= 16; shared memory checked by the library)."""
    if M > 16:
        return []
    out = []
    for kb in (2, 4, 8):
        for st in (2, 3, 4, 6):
            if grid == "small" and st > 4:
                continue
            out.append(dict(path=sgr.SGR_PATH_W8S, k_blocks_per_stage=kb, stages=st))
    return out


def candidate_configs_w4(simt: bool, M: int, K: int, grid: str) -> list[dict]:
    """Launch configurations of the NVFP4-weight kernels (the library refuses
    what does not fit)."""
    out = []
    if simt:
        if K % 32 or K > 7168:
            return []
        for cps in (1, 2, 3):
            for rps in (1, 2, 4):
                for st in (2, 4, 8):
                    if grid == "small" and st == 8:
                        continue
                    out.append(dict(path=sgr.SGR_PATH_SIMT, ctas_per_sm=cps, rows_per_stage=rps, stages=st))
        return out
    for kb in (4, 8):
        for st in (2, 3, 4, 6):
            if grid == "small" and st > 4:
                continue
            out.append(dict(path=sgr.SGR_PATH_W8, k_blocks_per_stage=kb, stages=st))
    return out


def candidate_configs_w8(simt: bool, M: int, K: int, grid: str) -> list[dict]:
    """Launch configurations of the FP8-weight kernels (shared memory checked
    by the library, which refuses what does not fit)."""
    out = []
    if simt:
        if M > 8 or K % 16:
            return []
        for cps in (1, 2, 3):
            for rps in (1, 2, 4):
                for st in (2, 4, 6, 8):
                    if grid == "small" and st not in (4, 6):
                        continue
                    out.append(dict(path=sgr.SGR_PATH_SIMT, ctas_per_sm=cps, rows_per_stage=rps, stages=st))
        return out
    if M > 256:
        return []
    for rb in (0, 64):
        for kb in (2, 4, 8):
            for st in (2, 3, 4, 6):
                for sa in (2, 3):
                    if grid == "small" and (st > 3 or sa > 2):
                        continue
                    out.append(dict(path=sgr.SGR_PATH_W8, k_blocks_per_stage=kb, stages=st, prefetch_stages=sa,
                                    rows_per_stage=rb))
    return out


def candidate_configs(path: int, M: int, K: int, grid: str) -> list[dict]:
    out = []
    if path == sgr.SGR_PATH_SIMT:
        if M > 16:
            return []
        for cps in (1, 2, 3):
            for rps in (1, 2, 4):
                for st in (2, 3, 4, 6, 8, 12, 16):
                    smem = 2048 + st * rps * K * 2
                    if smem * cps > 227 * 1024 or smem > 232448 or (cps == 3 and M > 2):
                        continue
                    if grid == "small" and st not in (4, 8, 12):
                        continue
                    out.append(dict(path=path, ctas_per_sm=cps, rows_per_stage=rps, stages=st))
    elif path == sgr.SGR_PATH_TC_ROWS:
        if M > 256:
            return []
        nt = (M + 15) // 16 * 16
        # slab height: N / SMs (48 at N = 7168), or 32 rows (two CTAs per SM)
        for rb, cfg_rb in ((48, 0), (32, 32)):
            for kb in (1, 2, 4, 8):
                for st in (2, 3, 4, 5, 6, 8, 10, 12):
                    slack = max(0, 16384 - rb * 128 - st * kb * nt * 128)
                    smem = 2048 + st * kb * (rb * 128 + nt * 128) + slack
                    if smem > 232448 or (cfg_rb and (M > 16 or smem > 113 * 1024)):
                        continue
                    if grid == "small" and st not in (2, 3, 4, 6):
                        continue
                    for pf in sorted({st, max(1, st - 1), max(1, st - 2)}):
                        out.append(dict(path=path, ctas_per_sm=1, k_blocks_per_stage=kb, stages=st,
                                        prefetch_stages=pf, rows_per_stage=cfg_rb))
        # 2-CTA K split (a slab per cluster, each CTA half of K): slabs of
        # N / (SMs / 2) rows, 16-64-token tiles
        if nt <= 64:
            for kb in (4, 8):
                for st in (2, 3, 4, 5, 6):
                    if grid == "small" and st not in (2, 3, 4):
                        continue
                    for pf in sorted({st, max(1, st - 1), max(1, st - 2)}):
                        out.append(dict(path=path, ctas_per_sm=1, k_blocks_per_stage=kb, stages=st,
                                        prefetch_stages=pf, rows_per_stage=0, k_split=2))
    elif path == sgr.SGR_PATH_TILE:
        if M < 32:
            return []
        for nt in (64, 128, 192, 256):
            for kb in (1, 2, 4):
                stage = kb * (128 * 128 + nt * 128)
                deepest = (232448 - 2048) // stage
                for st in range(2, min(deepest, 16) + 1):
                    if grid == "small" and st < deepest - 2:
                        continue
                    for pf in sorted({st, max(1, st - 1)}):
                        for split in (1, 2, 3, 4):
                            if (split == 2 and nt > 192) or (split == 3 and nt != 192) or (split == 4 and nt == 64):
                                continue
                            out.append(dict(path=path, ctas_per_sm=1, tile_n=nt, k_blocks_per_stage=kb, stages=st,
                                            prefetch_stages=pf, k_split=split))
    elif path == sgr.SGR_PATH_PAIR:
        if M < 32:
            return []
        for nt in (64, 96, 128, 192, 256):
            for kb in (1, 2, 4):
                stage = kb * (128 * 128 + (nt // 2) * 128)
                deepest = (232448 - 2048) // stage
                for st in range(2, min(deepest, 16) + 1):
                    if grid == "small" and st < deepest - 2:
                        continue
                    for pf in sorted({st, max(1, st - 1)}):
                        out.append(dict(path=path, ctas_per_sm=1, tile_n=nt, k_blocks_per_stage=kb, stages=st,
                                        prefetch_stages=pf))
    else:
        tiles = (M + 255) // 256
        nt = ((M + tiles - 1) // tiles + 15) // 16 * 16  # the library's token tile
        for kb in (1, 2, 4):
            for st in (2, 3, 4, 5, 6, 8, 12):
                for cps in (1, 2):
                    smem = 2048 + st * kb * (16384 + nt * 128)
                    if smem * cps > 228 * 1024 or smem > 232448:
                        continue
                    if grid == "small" and st not in (2, 4, 6):
                        continue
                    out.append(dict(path=path, ctas_per_sm=cps, k_blocks_per_stage=kb, stages=st))
    return out


FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}


def load_peaks(path: str | None = None) -> tuple[dict, str]:
    """HBM copy bandwidth (GB/s) and BF16 tensor throughput (TFLOP/s) measured
    on this GPU model (MEASURED_PEAKS.json at the repository root), else the
    fallback figures; returns (peaks, "measured" | "fallback")."""
    path = path or os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"])}, "measured"
    except (OSError, KeyError, ValueError, TypeError):
        return dict(FALLBACK_PEAKS), "fallback"


def build_row(M: int, N: int, K: int, backend: str, cfg: dict, copies: int, meta: dict, samples,
              peaks: dict, peak_source: str) -> dict:
    """One sweep row: timing statistics, achieved GB/s of algorithmic bytes
    (BF16: W, A, R, Y once; FP8 weights: codes, scales, A, R, Y once), TFLOP/s
    (2*M*N*K) and both as fractions of the peaks; or the error of a refused
    configuration (`samples` a string)."""
    row = {"m": M, "n": N, "k": K, "backend": backend, "config": cfg, "num_buffers": copies, **meta}
    if isinstance(samples, str):
        row.update({"valid": False, "error": samples})
        return row
    st = summarize(samples)
    row.update(st)
    if backend.startswith("w8"):
        nbytes = N * K + 4 * N + 2 * M * K + 4 * M * N
    elif backend.startswith("w4"):
        nbytes = N * K // 2 + N * ((K + 15) // 16) + 2 * M * K + 4 * M * N
    else:
        nbytes = 2 * (N * K + M * K + 2 * M * N)
    sec = st["median_us"] * 1e-6
    row["gbs"] = nbytes / sec / 1e9
    row["tflops"] = 2.0 * M * N * K / sec / 1e12
    row["frac_of_hbm_peak"] = row["gbs"] / peaks["hbm_gbs"]
    row["frac_of_tensor_peak"] = row["tflops"] / peaks["bf16_tflops"]
    row["peak_source"] = peak_source
    return row


def row_key(m: int, n: int, k: int, backend: str, cfg: dict) -> tuple:
    """Identity of a sweep row: shape, backend and launch configuration."""
    return (int(m), int(n), int(k), backend, json.dumps(cfg, sort_keys=True))


def load_done(path: str) -> set:
    """Keys of the rows already in a sweep output file (a missing file has
    none; a line cut short by an interrupted run is ignored)."""
    done = set()
    try:
        with open(path) as f:
            for line in f:
                try:
                    r = json.loads(line)
                    done.add(row_key(r["m"], r["n"], r["k"], r["backend"], r["config"]))
                except (ValueError, KeyError, TypeError):
                    continue
    except OSError:
        pass
    return done


def open_output(path: str, resume: bool):
    """The output file, appended to when resuming (after a newline if an
    interrupted run left the last line unfinished), else truncated."""
    if not resume:
        return open(path, "w")
    tail = b""
    try:
        with open(path, "rb") as f:
            f.seek(0, 2)
            if f.tell() > 0:
                f.seek(-1, 2)
                tail = f.read(1)
    except OSError:
        pass
    out = open(path, "a")
    if tail and tail != b"\n":
        out.write("\n")
    return out


def summarize(samples):
    ordered = sorted(samples)

    def pct(f):
        pos = f * (len(ordered) - 1)
        lo, hi = math.floor(pos), math.ceil(pos)
        if lo == hi:
            return ordered[lo]
        return ordered[lo] * (1 - (pos - lo)) + ordered[hi] * (pos - lo)

    mean = statistics.mean(samples)
    return {"median_us": statistics.median(samples), "p10_us": pct(0.1), "p90_us": pct(0.9),
            "mean_us": mean, "cv_pct": statistics.pstdev(samples) / mean * 100.0}


def graph_samples(launch, copies, stream, repeats: int, replays: int):
    """Eager call per copy, one graph holding all copies, warm replays, then
    `repeats` event-timed batches of `replays` replays: us per call."""
    with torch.cuda.stream(stream):
        for c in range(copies):
            launch(c)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for c in range(copies):
            launch(c)
    out = []
    with torch.cuda.stream(stream):
        for _ in range(10):
            g.replay()
        for _ in range(repeats):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(replays):
                g.replay()
            e1.record(stream)
            e1.synchronize()
            out.append(e0.elapsed_time(e1) * 1000.0 / (replays * copies))
    del g
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--m", type=int, nargs="+", default=[1, 2, 4, 8, 16])
    ap.add_argument("--n", type=int, default=inputs.N_LATENT_MOE)
    ap.add_argument("--k", type=int, default=inputs.K_LATENT_MOE)
    ap.add_argument("--paths", default="simt,tc,rows,tile")
    ap.add_argument("--grid", choices=("small", "full"), default="full")
    ap.add_argument("--copies", type=int, default=4)
    ap.add_argument("--repeats", type=int, default=7)
    ap.add_argument("--replays", type=int, default=50)
    ap.add_argument("--no-cublas", action="store_true")
    ap.add_argument("--config", action="append", default=[],
                    help="time only this configuration (JSON object of sgr_config fields; repeatable)")
    ap.add_argument("--output", default=None)
    ap.add_argument("--resume", action="store_true", help="append to --output, skipping rows already in it")
    args = ap.parse_args(argv)
    if args.resume and not args.output:
        ap.error("--resume needs --output")
    torch.cuda.set_device(0)
    sgr.sgr_init(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device=dev)
    N, K = args.n, args.k
    Ws = [inputs.make_weights(N, K, seed=s).to(dev) for s in range(args.copies)]
    props = torch.cuda.get_device_properties(dev)
    meta = {"device": props.name, "sms": props.multi_processor_count,
            "l2_bytes": props.L2_cache_size, "torch": torch.__version__}
    peaks, peak_source = load_peaks()
    done = load_done(args.output) if args.resume else set()
    out = open_output(args.output, args.resume) if args.output else None
    paths = {"simt": sgr.SGR_PATH_SIMT, "tc": sgr.SGR_PATH_TC, "rows": sgr.SGR_PATH_TC_ROWS,
             "tile": sgr.SGR_PATH_TILE, "pair": sgr.SGR_PATH_PAIR, "w8": sgr.SGR_PATH_W8, "w8simt": sgr.SGR_PATH_SIMT,
             "w8s": sgr.SGR_PATH_W8S, "w4": sgr.SGR_PATH_W8, "w4simt": sgr.SGR_PATH_SIMT}
    fp8 = [name for name in args.paths.split(",") if name in ("w8", "w8simt", "w8s")]
    if fp8:  # per-column-quantised E4M3 copies of the same weights
        q = [inputs.make_problem_w8(1, N, K, seed=s) for s in range(args.copies)]
        Wqs = [x.Wq.to(dev) for x in q]
        Scs = [x.scale.to(dev) for x in q]
    if any(name in ("w4", "w4simt") for name in args.paths.split(",")):  # NVFP4-quantised copies
        q4 = [inputs.make_problem_w4(1, N, K, seed=s) for s in range(args.copies)]
        W4s = [x.Wq4.to(dev) for x in q4]
        B4s = [x.bs.to(dev) for x in q4]
        G4s = [x.gs for x in q4]
    for M in args.m:
        A = inputs.make_rows(M, K, seed=10_000 + M).to(dev)
        Rs = [inputs.make_rows(M, N, seed=20_000 + 100 * M + s).to(dev) for s in range(args.copies)]
        Ys = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(args.copies)]
        rows = []

        def record(backend, cfg, samples):
            row = build_row(M, N, K, backend, cfg, args.copies, meta, samples, peaks, peak_source)
            if out:
                out.write(json.dumps(row, sort_keys=True) + "\n")
                out.flush()
            rows.append((backend, cfg, samples))

        if not args.no_cublas and row_key(M, N, K, "cublas_addmm", {}) not in done:
            launch = lambda c: torch.addmm(Rs[c], A, Ws[c].t(), out=Ys[c])
            record("cublas_addmm", {}, graph_samples(launch, args.copies, stream, args.repeats, args.replays))
        for name in args.paths.split(","):
            w8 = name in ("w8", "w8simt", "w8s")
            w4 = name in ("w4", "w4simt")
            if args.config:
                cands = [dict(json.loads(c), path=paths[name]) for c in args.config]
            elif w4:
                cands = candidate_configs_w4(name == "w4simt", M, K, args.grid)
            elif name == "w8s":
                cands = candidate_configs_w8s(M, args.grid)
            elif w8:
                cands = candidate_configs_w8(name == "w8simt", M, K, args.grid)
            else:
                cands = candidate_configs(paths[name], M, K, args.grid)
            backend = {"w8": "w8", "w8simt": "w8_simt", "w8s": "w8s", "w4": "w4", "w4simt": "w4_simt"}.get(name, name)
            for cfg in cands:
                if row_key(M, N, K, backend, cfg) in done:
                    continue
                c = sgr.make_config(**cfg)
                if w8:
                    launch = lambda i, c=c: sgr.skinny_gemm_residual_w8(A, Wqs[i], Scs[i], Rs[i], Ys[i], stream=stream,
                                                                       config=c)
                elif w4:
                    launch = lambda i, c=c: sgr.skinny_gemm_residual_w4(A, W4s[i], B4s[i], G4s[i], Rs[i], Ys[i],
                                                                       stream=stream, config=c)
                else:
                    launch = lambda i, c=c: sgr.skinny_gemm_residual_ex(A, Ws[i], Rs[i], Ys[i], stream=stream,
                                                                        config=c)
                try:
                    samples = graph_samples(launch, args.copies, stream, args.repeats, args.replays)
                except sgr.SgrError as e:
                    samples = str(e)
                record(backend, cfg, samples)
        best = {}
        for backend, cfg, samples in rows:
            if isinstance(samples, str):
                continue
            med = statistics.median(samples)
            if backend not in best or med < best[backend][0]:
                best[backend] = (med, cfg)
        print(f"M={M}: " + "; ".join(f"{b} {v[0]:.2f} us {v[1]}" for b, v in best.items()), flush=True)
    assert sgr.sgr_device_error() == 0
    return 0


if __name__ == "__main__":
    sys.exit(main())
