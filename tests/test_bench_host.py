"""Host-side parts of the benchmark that need no GPU: the reference arm's JSON
line (the CPU oracle timed on a bounded sample, same metric and workload as
the GPU arm) and the rule that a committed DRAM-traffic figure counts only
while the kernel's sources are the ones it was captured on."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_reference_arm_json_line():
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3", "--ref-budget", "2"], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == bench.workload_name(bench.M_LIST)  # the GPU arm's workload
    assert (d["steps"], d["warmup"], d["n_gpus"]) == (3, 3, 1)
    assert d["value"] > 0 and d["ms_per_step"] > 0
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] == d["value"] and cpu["cores"] >= 1 and cpu["sample"]
    assert cpu["cpu_model"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_committed_traffic_follows_the_source_digest(tmp_path, monkeypatch):
    kernel = "rows_skinny_kernel"
    csrc = tmp_path / "skinny_bf16_gemm_residual_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in bench.KERNEL_SOURCES[kernel]:
        (csrc / name).write_text("first version of " + name)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    digest = bench.kernel_source_digest(kernel)
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / f"{kernel}_traffic.md").write_text(
        f"# traffic\n\n- source_digest: `{digest}`\n- dram_bytes_per_launch: `51803648`\n")
    assert bench.committed_traffic(kernel) == pytest.approx(51803648.0)
    (csrc / bench.KERNEL_SOURCES[kernel][0]).write_text("changed")
    assert bench.committed_traffic(kernel) is None  # kernel changed since the capture
    assert bench.committed_traffic("no_such_kernel") is None


def test_algorithmic_bytes_and_ridge():
    assert bench.alg_bytes(1) == 2 * (7168 * 3584 + 3584 + 2 * 7168)
    assert bench.alg_flops(16) == 2 * 16 * 7168 * 3584
    peaks = {"hbm_gbs": 6772.9, "bf16_tflops": 1900.0}
    assert not bench.tensor_bound(16, peaks) and not bench.tensor_bound(128, peaks)
    assert bench.tensor_bound(1024, peaks)


def test_cpu_oracle_rate_single_and_all_threads():
    """The CPU baseline's two legs on a small slice of the workload: all host
    threads and one thread, each within its time budget."""
    from skinny_bf16_gemm_residual_gb300 import inputs

    Ws = [inputs.make_weights(64, 256, seed=s) for s in range(2)]
    per_m = {M: {"A_cpu": inputs.make_rows(M, 256, seed=M),
                 "R_cpu": [inputs.make_rows(M, 64, seed=100 + M + s) for s in range(2)]} for M in (1, 4)}
    old = (bench.N_DIM, bench.K_DIM)
    try:
        bench.N_DIM, bench.K_DIM = 64, 256
        rate, threads, desc, secs = bench.cpu_oracle_rate(Ws, per_m, (1, 4), 0.2)
        rate1, threads1, _, secs1 = bench.cpu_oracle_rate(Ws, per_m, (1, 4), 0.2, threads=1)
    finally:
        bench.N_DIM, bench.K_DIM = old
    assert threads == (os.cpu_count() or 1) and threads1 == 1
    assert rate > 0 and rate1 > 0 and 0.2 <= secs < 5 and 0.2 <= secs1 < 5
    assert "threads" in desc
    assert bench.cpu_model()


def test_cpu_model_names():
    x86 = "processor\t: 0\nvendor_id\t: GenuineIntel\nmodel name\t: Intel(R) Xeon(R) Processor\n"
    assert bench.cpu_model(x86) == "Intel(R) Xeon(R) Processor"
    grace = "processor\t: 0\nBogoMIPS\t: 2000.00\nCPU implementer\t: 0x41\nCPU architecture: 8\nCPU part\t: 0xd4f\n"
    assert bench.cpu_model(grace).startswith("Arm Neoverse V2")
    other = "CPU implementer\t: 0x51\nCPU part\t: 0x001\n"
    assert "part 0x001" in bench.cpu_model(other)
    assert bench.cpu_model("")
