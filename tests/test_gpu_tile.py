"""GPU parity of the tile GEMM path (128-token x tile_n output tiles on
tcgen05, residual and output handled row per thread) against the CPU oracle."""
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
TILE = sgr.SGR_PATH_TILE


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    torch.cuda.set_device(0)
    sgr.sgr_init(0)
    sgr.sgr_device_error(0, clear=True)
    yield
    assert sgr.sgr_device_error(0) == 0, "a kernel reported a timed-out wait"


def run_tile(p, **cfg):
    A, W, R = (t.cuda() for t in (p.A, p.W, p.R))
    Y = torch.full_like(R, float("nan"))
    sgr.skinny_gemm_residual_ex(A, W, R, Y, config=sgr.make_config(path=TILE, **cfg))
    torch.cuda.synchronize()
    return bits(Y)


# Ragged in every dimension: M below, at and across the 128-token tile; N not
# a multiple of the tile width or of 64 columns; K not a multiple of the
# 64-wide K block, and K = 8 (a single partial block).
SMALL = [(1, 520, 264), (5, 304, 8), (100, 1024, 520), (128, 256, 64), (129, 392, 1000),
         (250, 264, 1000), (300, 392, 264), (383, 1000, 136), (512, 2056, 1800), (640, 776, 3584)]


@pytest.mark.parametrize("tile_n", [0, 64, 128, 192, 256])
@pytest.mark.parametrize("M,N,K", SMALL)
def test_tile_small_shapes(M, N, K, tile_n):
    p = inputs.make_problem(M, N, K, seed=M * 5 + N + K)
    compare(run_tile(p, tile_n=tile_n), oracle_full(p.A, p.W, p.R), f"tile {M}x{N}x{K} nt={tile_n}")


@pytest.mark.parametrize("M", [32, 64, 128])
def test_tile_full_size_transition(M):
    p = inputs.make_problem(M, N_FULL, K_FULL, seed=M + 1)
    compare(run_tile(p), oracle_full(p.A, p.W, p.R), f"tile M={M}")


@pytest.mark.parametrize("M", [256, 512, 1024, 1000])
def test_tile_full_size_compute_bound_every_element(M):
    """The compute-bound sweep at the latent-MoE shape: every output element
    against the oracle."""
    p, ref = oracle_problem(M, N_FULL, K_FULL, seed=M)
    m = compare(run_tile(p), ref, f"tile M={M}")
    assert m["cosine"] > 0.999


def test_tile_full_size_every_tile_corner():
    """M = 1024: the corner elements of every 128 x 192 output tile (the
    library's choice of tile width at this size), of every epilogue warp's
    32-row block and of every 64-column group."""
    M = 1024
    p = inputs.make_problem(M, N_FULL, K_FULL, seed=9)
    got = run_tile(p, tile_n=192)
    rows = sorted({r for m0 in range(0, M, 128) for r in (m0, m0 + 31, m0 + 32, m0 + 127) if r < M})
    cols = sorted({c for n0 in range(0, N_FULL, 64) for c in (n0, n0 + 63) if c < N_FULL})
    ms, ns = np.meshgrid(rows, cols, indexing="ij")
    ms, ns = ms.ravel(), ns.ravel()
    ref = oracle.load().sample(p.A, p.W, p.R, ms, ns)
    compare(got[ms, ns], ref, "tile corners")


SPLIT_CONFIGS = [
    dict(tile_n=64, k_split=2, stages=9),
    dict(tile_n=128, k_split=2, k_blocks_per_stage=2, stages=3),
    dict(tile_n=64, k_split=2, k_blocks_per_stage=4, stages=2),
    dict(tile_n=128, k_split=2, stages=7),
    dict(tile_n=128, k_split=2, stages=3, prefetch_stages=1),
    dict(tile_n=192, k_split=2, stages=5),
    dict(tile_n=192, k_split=2, stages=2),
    dict(tile_n=192, k_split=3, stages=5),
    dict(tile_n=192, k_split=3, k_blocks_per_stage=2, stages=2, prefetch_stages=1),
    dict(tile_n=128, k_split=4, stages=7),
    dict(tile_n=128, k_split=4, k_blocks_per_stage=2, stages=3),
    dict(tile_n=192, k_split=4, stages=5),
    dict(tile_n=256, k_split=4, stages=4),
    dict(tile_n=256, k_split=4, k_blocks_per_stage=2, stages=2),
]


def split_refused(K, cfg):
    """The planner's rule: every rank but the last takes ceil(k_blocks / S)
    K blocks rounded up to whole stages, and the last rank needs at least one."""
    S, kp = cfg.get("k_split", 1), cfg.get("k_blocks_per_stage", 1)
    kb = (K + 63) // 64
    chunk = ((kb + S - 1) // S + kp - 1) // kp * kp
    return kb - (S - 1) * chunk < 1


@pytest.mark.parametrize("cfg", SPLIT_CONFIGS, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
@pytest.mark.parametrize("M,N,K", [(1, 1024, 1032), (100, 2056, 72), (128, 1000, 136), (200, 1512, 3584),
                                   (256, 2056, 1000)])
def test_tile_split_k_cluster(cfg, M, N, K):
    """K split over a 2-, 3- or 4-CTA cluster, partial sums handed over
    through distributed shared memory and summed in rank order; K of 2 or 3
    K blocks (a rank with a single block, or none: refused) and ragged M and
    N."""
    p = inputs.make_problem(M, N, K, seed=3 * M + K)
    if split_refused(K, cfg):  # the last rank would get no K block
        with pytest.raises(sgr.SgrError) as e:
            run_tile(p, **cfg)
        assert e.value.status == sgr.SGR_ERR_UNSUPPORTED
        return
    compare(run_tile(p, **cfg), oracle_full(p.A, p.W, p.R), f"tile split M={M} N={N} K={K} {cfg}")


@pytest.mark.parametrize("M", [32, 128, 256])
def test_tile_split_full_size(M):
    p = inputs.make_problem(M, N_FULL, K_FULL, seed=M + 5)
    got = run_tile(p, tile_n=128 if M <= 128 else 192, k_split=2)
    compare(got, oracle_full(p.A, p.W, p.R), f"tile split M={M}")


@pytest.mark.parametrize("tile_n,k_split", [(192, 3), (256, 4), (128, 4)])
@pytest.mark.parametrize("M", [32, 64, 100, 128])
def test_tile_wide_split_full_size_every_element(M, tile_n, k_split):
    """3- and 4-way K splits at the latent-MoE shape (38 x 3 or 28 x 4 CTAs),
    every element against the oracle.  A split whose clusters do not all fit
    on the device at once (56 four-CTA clusters at tile_n = 128) is refused."""
    p, ref = oracle_problem(M, N_FULL, K_FULL, seed=M + 6)
    try:
        got = run_tile(p, tile_n=tile_n, k_split=k_split)
    except sgr.SgrError as e:
        assert e.status == sgr.SGR_ERR_UNSUPPORTED and (N_FULL + tile_n - 1) // tile_n > 36
        return
    compare(got, ref, f"tile split {k_split} M={M} nt={tile_n}")


@pytest.mark.parametrize("cfg", [dict(tile_n=128, k_split=2), dict(tile_n=192, k_split=3), dict(tile_n=256, k_split=4)],
                         ids=lambda c: f"nt{c['tile_n']}-s{c['k_split']}")
def test_tile_split_strided_in_place_and_deterministic(cfg):
    M, N, K = 150, 1024, 1032
    p = inputs.make_problem(M, N, K, seed=57)
    Abig = torch.zeros((M, K + 136), dtype=torch.bfloat16, device="cuda")
    A = Abig[:, 64:64 + K]
    A.copy_(p.A)
    big = torch.full((M, N + 512), 3.0, dtype=torch.bfloat16, device="cuda")
    RY = big[:, 256:256 + N]
    RY.copy_(p.R)
    sgr.skinny_gemm_residual_ex(A, p.W.cuda(), RY, RY, config=sgr.make_config(path=TILE, **cfg))
    torch.cuda.synchronize()
    compare(bits(RY), oracle_full(p.A, p.W, p.R), "tile split strided in-place")
    assert torch.all(big[:, :256] == 3.0) and torch.all(big[:, 256 + N:] == 3.0)
    y1, y2 = run_tile(p, **cfg), run_tile(p, **cfg)
    assert np.array_equal(y1, y2) and np.array_equal(y1, bits(RY))


def test_tile_split_rejects():
    p = inputs.make_problem(300, 256, 256, seed=2)
    A, W, R = (t.cuda() for t in (p.A, p.W, p.R))
    for cfg in (dict(tile_n=256, k_split=2), dict(tile_n=128, k_split=3), dict(tile_n=64, k_split=-1),
                dict(tile_n=64, k_split=3), dict(tile_n=64, k_split=4), dict(tile_n=256, k_split=3),
                dict(tile_n=192, k_split=5)):
        with pytest.raises(sgr.SgrError) as e:
            sgr.skinny_gemm_residual_ex(A, W, R, config=sgr.make_config(path=TILE, **cfg))
        assert e.value.status == sgr.SGR_ERR_UNSUPPORTED, cfg
    q = inputs.make_problem(4, 256, 8, seed=3)  # a single K block cannot be split
    with pytest.raises(sgr.SgrError) as e:
        sgr.skinny_gemm_residual_ex(q.A.cuda(), q.W.cuda(), q.R.cuda(),
                                    config=sgr.make_config(path=TILE, tile_n=64, k_split=2))
    assert e.value.status == sgr.SGR_ERR_UNSUPPORTED
    big = inputs.make_problem(1024, N_FULL, 64, seed=4)  # 304 tiles: more than one per cluster
    with pytest.raises(sgr.SgrError) as e:
        sgr.skinny_gemm_residual_ex(big.A.cuda(), big.W.cuda(), big.R.cuda(),
                                    config=sgr.make_config(path=TILE, tile_n=192, k_split=2))
    assert e.value.status == sgr.SGR_ERR_UNSUPPORTED


TILE_CONFIGS = [
    dict(tile_n=64, stages=2),
    dict(tile_n=64, stages=9),
    dict(tile_n=128, stages=7, prefetch_stages=3),
    dict(tile_n=192, stages=5),
    dict(tile_n=256, stages=4),
    dict(tile_n=128, stages=3, prefetch_stages=1),
    dict(tile_n=128, stages=6),
    dict(tile_n=192, stages=2),
    dict(tile_n=192, stages=4, prefetch_stages=2),
    dict(tile_n=256, stages=3),
    dict(tile_n=256, stages=2, prefetch_stages=1),
    dict(tile_n=128, k_blocks_per_stage=2, stages=3),
    dict(tile_n=192, k_blocks_per_stage=2, stages=2, prefetch_stages=1),
    dict(tile_n=64, k_blocks_per_stage=4, stages=2),
]


@pytest.mark.parametrize("cfg", TILE_CONFIGS, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
@pytest.mark.parametrize("M", [1, 200, 700])
def test_tile_configs(cfg, M):
    N, K = 2056, 1032
    p = inputs.make_problem(M, N, K, seed=13 + M)
    compare(run_tile(p, **cfg), oracle_full(p.A, p.W, p.R), f"tile M={M} {cfg}")


def test_tile_rejects_bad_config():
    p = inputs.make_problem(300, 256, 256, seed=1)
    A, W, R = (t.cuda() for t in (p.A, p.W, p.R))
    for cfg in (dict(tile_n=96), dict(tile_n=320), dict(tile_n=32), dict(ctas_per_sm=2),
                dict(tile_n=256, stages=5), dict(tile_n=64, stages=3, prefetch_stages=4), dict(stages=17),
                dict(token_tile=64), dict(k_blocks_per_stage=3), dict(tile_n=256, k_blocks_per_stage=4, stages=2)):
        with pytest.raises(sgr.SgrError) as e:
            sgr.skinny_gemm_residual_ex(A, W, R, config=sgr.make_config(path=TILE, **cfg))
        assert e.value.status == sgr.SGR_ERR_UNSUPPORTED, cfg


def test_tile_integer_inputs_exact():
    M, N, K = 300, 1024, 1024
    A = inputs.integer_bf16((M, K), -2, 2, 14)
    W = inputs.integer_bf16((N, K), -2, 2, 15)
    R = inputs.integer_bf16((M, N), -8, 8, 16)
    want = A.to(torch.int64) @ W.to(torch.int64).T + R.to(torch.int64)
    assert want.abs().max() < 2 ** 24  # every FP32 partial sum is an exact integer
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    sgr.skinny_gemm_residual_ex(A.cuda(), W.cuda(), R.cuda(), Y, config=sgr.make_config(path=TILE))
    torch.cuda.synchronize()
    assert np.array_equal(bits(Y), bits(want.to(torch.bfloat16)))


def test_tile_deterministic_and_pdl_off():
    p = inputs.make_problem(384, 2048, 1536, seed=44)
    y1 = run_tile(p)
    y2 = run_tile(p)
    A, W, R = (t.cuda() for t in (p.A, p.W, p.R))
    Y3 = torch.empty_like(R)
    sgr.skinny_gemm_residual_ex(A, W, R, Y3, flags=sgr.SGR_FLAG_NO_PDL, config=sgr.make_config(path=TILE))
    torch.cuda.synchronize()
    assert np.array_equal(y1, y2) and np.array_equal(y1, bits(Y3))


def test_tile_strided_column_slices_and_in_place():
    """A is a column slice of a wider buffer; R and Y are the same column slice
    of a wider [M, hidden] buffer (in-place residual update); columns outside
    the slice are untouched."""
    M, N, K = 260, 1024, 1032
    p = inputs.make_problem(M, N, K, seed=56)
    Abig = torch.zeros((M, K + 136), dtype=torch.bfloat16, device="cuda")
    A = Abig[:, 64:64 + K]
    A.copy_(p.A)
    big = torch.full((M, N + 512), 3.0, dtype=torch.bfloat16, device="cuda")
    RY = big[:, 256:256 + N]
    RY.copy_(p.R)
    sgr.skinny_gemm_residual_ex(A, p.W.cuda(), RY, RY, config=sgr.make_config(path=TILE))
    torch.cuda.synchronize()
    compare(bits(RY), oracle_full(p.A, p.W, p.R), "tile strided in-place")
    assert torch.all(big[:, :256] == 3.0) and torch.all(big[:, 256 + N:] == 3.0)


def test_tile_graph_replay_matches_eager():
    probs = [inputs.make_problem(512, 1024, 1024, seed=80 + s) for s in range(3)]
    dev = [[t.cuda() for t in (q.A, q.W, q.R)] for q in probs]
    outs = [torch.empty_like(d[2]) for d in dev]
    cfg = sgr.make_config(path=TILE)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for (A, W, R), Y in zip(dev, outs):
            sgr.skinny_gemm_residual_ex(A, W, R, Y, config=cfg)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = [bits(Y) for Y in outs]
    for Y in outs:
        Y.fill_(0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for (A, W, R), Y in zip(dev, outs):
            sgr.skinny_gemm_residual_ex(A, W, R, Y, config=cfg)
    for _ in range(10):
        g.replay()
    torch.cuda.synchronize()
    for e, Y in zip(eager, outs):
        assert np.array_equal(e, bits(Y))
    compare(eager[2], oracle_full(probs[2].A, probs[2].W, probs[2].R), "tile graph")
