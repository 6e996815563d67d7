"""GPU parity of the tensor-core (tcgen05) path against the CPU oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import skinny_bf16_gemm_residual_gb300 as sgr
from skinny_bf16_gemm_residual_gb300 import inputs
from parity import bits, compare, oracle_full, oracle_problem

import oracle

pytestmark = pytest.mark.gpu

N_FULL, K_FULL = inputs.N_LATENT_MOE, inputs.K_LATENT_MOE
TC = sgr.SGR_PATH_TC


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    torch.cuda.set_device(0)
    sgr.sgr_init(0)
    sgr.sgr_device_error(0, clear=True)
    yield
    assert sgr.sgr_device_error(0) == 0, "a kernel reported a timed-out wait"


ROWS = sgr.SGR_PATH_TC_ROWS


def run_tc(p, path=TC, **cfg):
    A, W, R = (t.cuda() for t in (p.A, p.W, p.R))
    Y = torch.full_like(R, float("nan"))
    sgr.skinny_gemm_residual_ex(A, W, R, Y, config=sgr.make_config(path=path, **cfg))
    torch.cuda.synchronize()
    return bits(Y)


SMALL = [(1, 520, 264), (3, 7168, 64), (4, 2056, 3584), (5, 304, 8), (7, 1512, 1800),
         (16, 2056, 3584), (16, 8, 3584), (1, 8, 8), (13, 152, 1792), (17, 200, 136),
         (40, 1000, 1032), (100, 1024, 520), (250, 264, 1000), (300, 392, 264)]


PATHS = pytest.mark.parametrize("path", [TC, ROWS], ids=["streamk", "rows"])


@PATHS
@pytest.mark.parametrize("M,N,K", SMALL)
def test_tc_small_shapes(M, N, K, path):
    p = inputs.make_problem(M, N, K, seed=M * 7 + N + K)
    if path == ROWS and M > 256:  # the row-slab kernel holds at most 256 tokens
        with pytest.raises(sgr.SgrError) as e:
            run_tc(p, path)
        assert e.value.status == sgr.SGR_ERR_UNSUPPORTED
        return
    compare(run_tc(p, path), oracle_full(p.A, p.W, p.R), f"path {path} {M}x{N}x{K}")


@PATHS
@pytest.mark.parametrize("M", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_tc_full_size_m_sweep(M, seed, path):
    p = inputs.make_problem(M, N_FULL, K_FULL, seed=seed)
    compare(run_tc(p, path), oracle_full(p.A, p.W, p.R), f"path {path} M={M} seed={seed}")


@PATHS
@pytest.mark.parametrize("M", [32, 64, 128])
def test_tc_full_size_transition(M, path):
    p = inputs.make_problem(M, N_FULL, K_FULL, seed=M)
    compare(run_tc(p, path), oracle_full(p.A, p.W, p.R), f"path {path} M={M}")


ROWS_CONFIGS = [
    dict(k_blocks_per_stage=1, stages=2),
    dict(k_blocks_per_stage=1, stages=8),
    dict(k_blocks_per_stage=2, stages=5),
    dict(k_blocks_per_stage=4, stages=3),
    dict(k_blocks_per_stage=8, stages=2),
    dict(k_blocks_per_stage=3, stages=4),
    dict(k_blocks_per_stage=2, stages=3, token_tile=64),
    dict(k_blocks_per_stage=8, stages=3, prefetch_stages=1),
    dict(k_blocks_per_stage=8, stages=3, prefetch_stages=3),
    dict(k_blocks_per_stage=4, stages=4, prefetch_stages=2),
    dict(rows_per_stage=32, k_blocks_per_stage=8, stages=2),
    dict(rows_per_stage=32, k_blocks_per_stage=4, stages=4, prefetch_stages=2),
    dict(rows_per_stage=24, k_blocks_per_stage=4, stages=3),
    dict(rows_per_stage=64, k_blocks_per_stage=4, stages=3),
    dict(rows_per_stage=8, k_blocks_per_stage=8, stages=3),
]


@pytest.mark.parametrize("cfg", ROWS_CONFIGS, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
@pytest.mark.parametrize("M", [1, 9, 16])
def test_rows_configs(cfg, M):
    p = inputs.make_problem(M, N_FULL, K_FULL, seed=71 + M)
    compare(run_tc(p, ROWS, **cfg), oracle_full(p.A, p.W, p.R), f"rows M={M} {cfg}")


def test_rows_rejects_bad_config():
    p = inputs.make_problem(20, 256, 256, seed=1)
    A, W, R = (t.cuda() for t in (p.A, p.W, p.R))
    for cfg in (dict(token_tile=16), dict(ctas_per_sm=2), dict(k_blocks_per_stage=8, stages=12),
                dict(stages=2, prefetch_stages=3), dict(rows_per_stage=20), dict(rows_per_stage=136)):
        with pytest.raises(sgr.SgrError) as e:
            sgr.skinny_gemm_residual_ex(A, W, R, config=sgr.make_config(path=ROWS, **cfg))
        assert e.value.status == sgr.SGR_ERR_UNSUPPORTED


@pytest.mark.parametrize("M", [256, 512, 1024])
def test_tc_full_size_compute_bound_every_element(M):
    """The stream-K kernel on the compute-bound sweep: every output element."""
    p, ref = oracle_problem(M, N_FULL, K_FULL, seed=M)
    compare(run_tc(p), ref, f"tc M={M}")


TC_CONFIGS = [
    dict(k_blocks_per_stage=1, stages=4),
    dict(k_blocks_per_stage=1, stages=8),
    dict(k_blocks_per_stage=2, stages=3),
    dict(k_blocks_per_stage=4, stages=2),
    dict(k_blocks_per_stage=2, stages=2, ctas_per_sm=2),
    dict(k_blocks_per_stage=1, stages=3, token_tile=32),
    dict(k_blocks_per_stage=3, stages=3),
]


@pytest.mark.parametrize("cfg", TC_CONFIGS, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
@pytest.mark.parametrize("M", [1, 8, 48])
def test_tc_configs(cfg, M):
    p = inputs.make_problem(M, N_FULL, K_FULL, seed=31 + M)
    compare(run_tc(p, **cfg), oracle_full(p.A, p.W, p.R), f"tc M={M} {cfg}")


def test_tc_integer_inputs_exact():
    M, N, K = 16, 2048, 1024
    A = inputs.integer_bf16((M, K), -2, 2, 4)
    W = inputs.integer_bf16((N, K), -2, 2, 5)
    R = inputs.integer_bf16((M, N), -8, 8, 6)
    want = A.to(torch.int64) @ W.to(torch.int64).T + R.to(torch.int64)
    assert want.abs().max() < 2 ** 24  # every FP32 partial sum is an exact integer
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    sgr.skinny_gemm_residual_ex(A.cuda(), W.cuda(), R.cuda(), Y, config=sgr.make_config(path=TC))
    torch.cuda.synchronize()
    assert np.array_equal(bits(Y), bits(want.to(torch.bfloat16)))


def test_tc_deterministic_across_runs_and_pdl():
    """Split-K partials are summed in K order, so repeated runs give the same bits."""
    p = inputs.make_problem(8, N_FULL, K_FULL, seed=44)
    y1 = run_tc(p)
    y2 = run_tc(p)
    A, W, R = (t.cuda() for t in (p.A, p.W, p.R))
    Y3 = torch.empty_like(R)
    sgr.skinny_gemm_residual_ex(A, W, R, Y3, flags=sgr.SGR_FLAG_NO_PDL, config=sgr.make_config(path=TC))
    torch.cuda.synchronize()
    assert np.array_equal(y1, y2) and np.array_equal(y1, bits(Y3))


def test_tc_strided_and_in_place():
    M, N, K = 6, 2048, 1024
    p = inputs.make_problem(M, N, K, seed=55)
    Abig = torch.zeros((M, K + 128), dtype=torch.bfloat16, device="cuda")
    A = Abig[:, 64:64 + K]
    A.copy_(p.A)
    RY = p.R.cuda().clone()
    sgr.skinny_gemm_residual_ex(A, p.W.cuda(), RY, RY, config=sgr.make_config(path=TC))
    torch.cuda.synchronize()
    compare(bits(RY), oracle_full(p.A, p.W, p.R), "tc strided in-place")


def test_tc_graph_replays_reuse_counters():
    """The split-K tile counters reset themselves: many graph replays of
    several calls keep giving the eager bits."""
    probs = [inputs.make_problem(4, N_FULL, K_FULL, seed=60 + s) for s in range(3)]
    dev = [[t.cuda() for t in (q.A, q.W, q.R)] for q in probs]
    outs = [torch.empty_like(d[2]) for d in dev]
    cfg = sgr.make_config(path=TC)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for (A, W, R), Y in zip(dev, outs):
            sgr.skinny_gemm_residual_ex(A, W, R, Y, config=cfg)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = [bits(Y) for Y in outs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for (A, W, R), Y in zip(dev, outs):
            sgr.skinny_gemm_residual_ex(A, W, R, Y, config=cfg)
    for _ in range(20):
        g.replay()
    torch.cuda.synchronize()
    for e, Y in zip(eager, outs):
        assert np.array_equal(e, bits(Y))
    compare(eager[1], oracle_full(probs[1].A, probs[1].W, probs[1].R), "tc graph")


def test_tc_rejects_bad_config():
    p = inputs.make_problem(4, 256, 256, seed=1)
    A, W, R = (t.cuda() for t in (p.A, p.W, p.R))
    for cfg in (dict(token_tile=24), dict(token_tile=512), dict(k_blocks_per_stage=4, stages=32),
                dict(ctas_per_sm=3)):
        with pytest.raises(sgr.SgrError) as e:
            sgr.skinny_gemm_residual_ex(A, W, R, config=sgr.make_config(path=TC, **cfg))
        assert e.value.status == sgr.SGR_ERR_UNSUPPORTED
