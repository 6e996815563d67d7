"""Launch-plan invariants checked on the CPU: the host planners of the
row-slab, FP8 row-slab and tile kernels (compiled with nvcc into a small host
program, tests/plan_probe.cu) are run over a grid of shapes and
configurations, and every accepted plan must fit the budgets the kernels rely
on: shared memory per CTA, tensor-memory columns, the barrier region, the MMA
window (128 rows, N <= 256), whole coverage of N and K, and room for the
epilogue's hand-over buffers in the drained rings."""
import json
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "skinny_bf16_gemm_residual_gb300", "csrc")
SMEM_LIMIT = 232448


@pytest.fixture(scope="module")
def plans(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path_factory.mktemp("plans") / "plan_probe")
    subprocess.run([nvcc, "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", f"-I{CSRC}",
                    f"-I{os.path.join(ROOT, 'include')}", os.path.join(ROOT, "tests", "plan_probe.cu"),
                    "-o", exe, "-lcuda"], check=True, capture_output=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    rows = [json.loads(line) for line in out.splitlines() if line.strip()]
    assert rows
    return rows


def test_row_slab_plans(plans):
    rows = [p for p in plans if p["kind"] == "rows"]
    assert len(rows) > 100 and sum(p["ksplit"] == 2 for p in rows) > 50
    for p in rows:
        assert p["smem"] <= SMEM_LIMIT, p
        assert p["RB"] % 8 == 0 and p["RB"] <= 128, p
        assert p["G"] * p["RB"] <= 128 and p["G"] * p["NT"] <= 256, p            # one MMA window
        assert p["kbps"] % p["G"] == 0, p
        assert p["NT"] >= p["M"] and p["NT"] % 16 == 0, p
        decode_epi = p["NT"] == 16 and p["G"] * p["RB"] <= 128
        # two MMA issuers (alternate windows, own accumulators) only under the
        # 16-token epilogues that add them, with two or more windows a stage
        assert p["issuers"] == (2 if decode_epi and p["kbps"] >= 2 * p["G"] else 1), p
        # kernel instance by epilogue family: 16-token tiles with up to two
        # and with three or four packed groups (224 threads, the only ones with
        # a second issuer), 64-token register form, the rest
        want_mode = (0 if p["G"] <= 2 else 3) if p["NT"] == 16 else (2 if p["NT"] == 64 and p["G"] <= 2 else 1)
        assert p["mode"] == want_mode, p
        assert p["threads"] == (224 if p["mode"] in (0, 3) else 192), p
        acc_cols = p["issuers"] * p["G"] * p["NT"]
        # the register epilogues' warm-up pass (16 tokens, and 32-64 tokens in
        # at most two groups) reads as many columns again, unwritten
        warm_epi = decode_epi or (p["NT"] in (32, 48, 64) and p["G"] <= 2 and p["G"] * p["RB"] <= 128)
        assert p["tmem_cols"] >= (2 if warm_epi else 1) * acc_cols and p["tmem_cols"] <= 512, p
        # alignment slack and barrier region, the rings, the MMA window's
        # over-read slack, and the 32-64-token warm-up pass's 512-byte scratch
        # (its exchange: up to NT + 4 floats)
        assert p["smem"] == 2048 + p["w_ring"] + p["a_ring"] + p["slack"] + (512 if p["NT"] > 16 else 0), p
        if warm_epi:
            assert (p["NT"] + 4) * 4 <= 512, p
        ks = p["ksplit"]
        slabs = p["grid"] // ks
        assert p["grid"] % ks == 0, p                                            # whole clusters
        assert slabs * p["RB"] >= p["N"] > (slabs - 1) * p["RB"], p             # every row, no empty slab
        assert ks * p["k_stages"] * p["kbps"] * 64 >= p["K"], p                  # both ranks cover K
        assert ks == 1 or (p["k_stages"] - 1) * p["kbps"] * 64 < p["K"], p      # rank 0 starts inside K
        if ks == 2:
            # the split's partial sums are completed in the 16-64-token
            # register epilogues (at most two groups), with two hand-over rows
            # per W row in the drained ring
            assert warm_epi and p["G"] <= 2 and p["mode"] in (0, 1, 2), p
            assert 2 * p["RB"] * (80 if p["NT"] == 16 else (p["NT"] + 4) * 4) <= p["w_ring"] + p["a_ring"], p
        assert 1 <= p["prefetch"] <= p["stages"], p
        # landing and slot-free barriers per stage, accumulator and drain
        # barriers, the TMEM address and the abort flag
        # and the K split's hand-over barrier (below the warm-up pass's
        # scratch at byte 960 of the region)
        assert (2 * p["stages"] + 3) * 8 + 8 <= 960, p
        drained = p["w_ring"] + p["a_ring"]
        # hand-over buffers of the epilogues live in the drained rings
        if p["NT"] == 16 and p["G"] <= 2:
            assert p["RB"] * 80 <= drained, p
        elif p["NT"] in (32, 48, 64) and p["G"] <= 2:
            assert p["RB"] * (p["NT"] + 4) * 4 <= drained, p
        else:
            assert p["G"] * p["RB"] * (p["NT"] + 4) * 4 <= drained, p


def test_fp8_row_slab_plans(plans):
    rows = [p for p in plans if p["kind"] == "w8"]
    assert len(rows) > 100 and sum(p["fp4"] for p in rows) > 50
    for p in rows:
        assert p["smem"] <= SMEM_LIMIT, p
        assert p["G"] * p["RB"] <= 128 and p["G"] * p["NT"] <= 256, p
        assert p["kbps"] % 2 == 0 and p["kbps"] % p["G"] == 0, p
        if p["fp4"]:
            # 256-code boxes (kbps/4 per stage) and the RB rows' block scales (kbps * 4 bytes each)
            # inside the stage, whose size keeps the next stage's boxes 1024-byte aligned
            assert p["kbps"] % 4 == 0, p
            assert p["w_stage"] % 1024 == 0 and p["w_stage"] >= p["kbps"] // 4 * p["RB"] * 128 + p["RB"] * p["kbps"] * 4, p
        else:
            assert p["w_stage"] == p["kbps"] // 2 * p["RB"] * 128, p
        wins = p["kbps"] // p["G"]
        assert p["tmem_cols"] in (256, 512), p
        assert p["acc_cols"] >= p["G"] * p["NT"], p
        assert p["slots"] >= 2 and p["acc_cols"] + p["slots"] * wins * 32 <= p["tmem_cols"], p
        barriers = (2 * p["stages"] + 2 * p["a_stages"] + 2 * p["slots"] + 3) * 8 + 8
        assert barriers <= 1024, p
        quarters = (p["G"] * p["RB"] + 31) // 32
        assert p["conv_warps"] == 2 * quarters and p["conv_warps"] <= 8, p
        assert p["grid"] * p["RB"] >= p["N"] > (p["grid"] - 1) * p["RB"], p
        assert p["k_stages"] * p["kbps"] * 64 >= p["K"], p
        assert p["rtile"] >= p["RB"] * p["NT"] * 2, p
        drained = p["w_ring"] + p["a_ring"]
        if p["NT"] == 16 and p["G"] <= 2:
            assert p["RB"] * 80 <= drained, p
        else:
            assert p["G"] * p["RB"] * (p["NT"] + 4) * 4 <= drained, p


def test_tile_plans(plans):
    rows = [p for p in plans if p["kind"] == "tile"]
    assert len(rows) > 50
    assert {p["split"] for p in rows} == {1, 2, 3, 4}, "every split width is planned somewhere on the grid"
    for p in rows:
        assert p["smem"] <= SMEM_LIMIT, p
        assert p["NT"] in (64, 128, 192, 256), p
        assert p["tmem_cols"] >= 2 * p["NT"] and p["tmem_cols"] <= 512, p       # two accumulators
        assert p["m_tiles"] * 128 >= p["M"] and p["n_tiles"] * p["NT"] >= p["N"], p
        assert p["k_blocks"] * 64 >= p["K"], p
        S = p["split"]
        if S > 1:
            assert 1 <= p["kb_split"] and (S - 1) * p["kb_split"] < p["k_blocks"], p  # every rank gets K blocks
            assert p["kb_split"] % p["kbps"] == 0, p
            assert p["grid"] == S * p["m_tiles"] * p["n_tiles"] <= 152, p         # one tile per cluster, one wave
            assert (p["NT"] // S) % 16 == 0 and p["NT"] % S == 0, p               # whole 16-column pieces per rank
            ring = p["stages"] * p["kbps"] * (128 * 128 + p["NT"] * 128)
            assert (S - 1) * 128 * (p["NT"] // S) * 4 <= ring, p                 # hand-over slots inside the ring
        else:
            assert p["grid"] == min(p["m_tiles"] * p["n_tiles"], 152), p


def test_pair_plans(plans):
    rows = [p for p in plans if p["kind"] == "pair"]
    assert len(rows) > 50
    for p in rows:
        assert p["smem"] <= SMEM_LIMIT, p
        assert p["NT"] in (64, 96, 128, 192, 256), p
        assert p["tmem_cols"] >= 2 * p["NT"] and p["tmem_cols"] <= 512, p       # two accumulators
        assert p["m_tiles"] * 256 >= p["M"] and p["n_tiles"] * p["NT"] >= p["N"], p
        assert p["k_blocks"] * 64 >= p["K"], p
        assert p["grid"] % 2 == 0 and p["grid"] == 2 * min(p["m_tiles"] * p["n_tiles"], 76), p
        # every box of a stage starts on a 1024-byte swizzle-atom boundary
        assert (128 * 128) % 1024 == 0 and (p["NT"] // 2 * 128) % 1024 == 0 and p["stage_bytes"] % 1024 == 0, p
        assert (2 * p["stages"] + 5) * 8 + 8 <= 1024, p                         # barrier region
        # the even CTA arms each stage with both CTAs' bytes: within the tx-count range
        assert 2 * p["stage_bytes"] < 2 ** 20, p


def test_fp8_split_plans(plans):
    rows = [p for p in plans if p["kind"] == "w8s"]
    assert len(rows) > 50 and {p["issuers"] for p in rows} == {1, 2}
    for p in rows:
        assert p["smem"] <= SMEM_LIMIT, p
        # alignment slack, barrier region, weight ring, operand span, warm-up scratch
        assert p["smem"] == 2048 + p["ring"] + p["span"] + 256, p
        assert p["span"] >= p["kbp"] * 2 * p["NT"] * 128 and p["span"] >= (128 - p["RB"]) * 128, p
        assert p["G"] * p["RB"] <= 128 and p["G"] * 2 * p["NT"] <= 256 and p["kbps"] % p["G"] == 0, p
        assert p["kbp"] % p["G"] == 0 and p["kb"] <= p["kbp"] < p["kb"] + p["G"], p
        assert p["k_stages"] * p["kbps"] >= p["kb"] and p["kb"] * 128 >= p["K"], p
        # a second MMA issuer needs two windows a stage and one in the first stage
        assert p["issuers"] == (2 if p["kbps"] >= 2 * p["G"] and p["kb"] > p["G"] else 1), p
        # one accumulator per issuer, as many columns again for the warm-up pass
        acc = p["issuers"] * p["G"] * 2 * p["NT"]
        assert 2 * acc <= p["tmem_cols"] <= 512 and p["tmem_cols"] & (p["tmem_cols"] - 1) == 0, p
        assert (2 * p["stages"] + p["k_stages"] + 2) * 8 + 8 <= 896, p       # barriers below the token words
        assert (p["G"] - 1) * p["RB"] * 80 <= p["ring"], p                   # epilogue hand-over in the drained ring
        assert p["grid"] * p["RB"] >= p["N"] > (p["grid"] - 1) * p["RB"], p


def test_large_ends_are_planned_or_refused(plans):
    """The largest K is planned by every kernel; N = 2^17 is refused by the
    row slabs (more than 128 rows per CTA on 152 SMs) and planned by the tile
    kernels, which also take M = 1024 (the row slabs hold at most 256 tokens)."""
    kinds = lambda **kw: {p["kind"] for p in plans if all(p[k] == v for k, v in kw.items())}  # noqa: E731
    assert kinds(K=1048576) == {"rows", "w8", "tile", "pair"}
    assert kinds(N=131072) == {"tile", "pair"}
    assert kinds(M=1024) == {"tile", "pair"}
    assert {"rows", "w8", "tile"} <= kinds(K=65536, M=256)


def test_row_slab_default_configurations(plans):
    """The default configuration of shapes without a table entry: a plan the
    kernel accepts, and the 2-CTA K split exactly for slabs of at most 32 rows
    over K >= 4096 at up to 64 tokens (where the split plan fits)."""
    rows = [p for p in plans if p["kind"] == "rows_default"]
    assert len(rows) > 40
    for p in rows:
        assert p["plan_ok"] == 1, p
        rb = -(-p["N"] // 152)
        rb = -(-rb // 8) * 8
        want = rb <= 32 and p["K"] >= 4096 and p["token_tile"] <= 64
        assert (p["k_split"] == 2) == want, p
        if want:  # the split's slab: N / 76 rows rounded up to 8
            assert p["RB"] == -(-(-(-p["N"] // 76)) // 8) * 8, p
    assert any(p["k_split"] == 2 for p in rows) and any(p["k_split"] == 0 for p in rows)

