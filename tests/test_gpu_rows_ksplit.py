"""GPU parity of the row-slab kernel with the 2-CTA K split (k_split = 2:
each W slab on a 2-CTA cluster, one CTA per half of K, the partial sums added
in the epilogue through distributed shared memory) against the CPU oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import skinny_bf16_gemm_residual_gb300 as sgr
from skinny_bf16_gemm_residual_gb300 import inputs
from parity import bits, compare, oracle_full

pytestmark = pytest.mark.gpu

ROWS = sgr.SGR_PATH_TC_ROWS
# The down-projection of the latent-MoE block (K = 7168 -> N = 3584), the
# shape the split is for, and the up-projection.
N_DOWN, K_DOWN = inputs.K_LATENT_MOE, inputs.N_LATENT_MOE
N_UP, K_UP = inputs.N_LATENT_MOE, inputs.K_LATENT_MOE


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    torch.cuda.set_device(0)
    sgr.sgr_init(0)
    sgr.sgr_device_error(0, clear=True)
    yield
    assert sgr.sgr_device_error(0) == 0, "a kernel reported a timed-out wait"


def run_split(p, flags=0, **cfg):
    A, W, R = (t.cuda() for t in (p.A, p.W, p.R))
    Y = torch.full_like(R, float("nan"))
    sgr.skinny_gemm_residual_ex(A, W, R, Y, flags=flags, config=sgr.make_config(path=ROWS, k_split=2, **cfg))
    torch.cuda.synchronize()
    return bits(Y)


# Ragged in every dimension: K of one partial block (rank 1 reads only the
# zero fill past K), K not a multiple of a stage, N not a multiple of the
# slab, a single slab, 1-64 tokens (16-token decode form, 32/48/64-token
# register forms).
SMALL = [(1, 520, 264), (5, 304, 8), (3, 8, 3584), (16, 2056, 3584), (17, 200, 136), (40, 1000, 1032),
         (64, 1024, 520), (33, 152, 1792), (48, 2056, 7168), (9, 4104, 7168)]


@pytest.mark.parametrize("M,N,K", SMALL)
def test_split_small_shapes(M, N, K):
    p = inputs.make_problem(M, N, K, seed=M * 11 + N + K)
    compare(run_split(p), oracle_full(p.A, p.W, p.R), f"split {M}x{N}x{K}")


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16, 17, 32, 48, 64])
def test_split_down_projection_every_element(M):
    p = inputs.make_problem(M, N_DOWN, K_DOWN, seed=500 + M)
    compare(run_split(p), oracle_full(p.A, p.W, p.R), f"split down M={M}")


@pytest.mark.parametrize("M", [1, 16, 64])
def test_split_up_projection_every_element(M):
    p = inputs.make_problem(M, N_UP, K_UP, seed=600 + M)
    compare(run_split(p), oracle_full(p.A, p.W, p.R), f"split up M={M}")


SPLIT_CONFIGS = [
    dict(k_blocks_per_stage=8, stages=3),
    dict(k_blocks_per_stage=8, stages=2, prefetch_stages=1),
    dict(k_blocks_per_stage=4, stages=4, prefetch_stages=2),
    dict(k_blocks_per_stage=2, stages=6),
    dict(k_blocks_per_stage=1, stages=8),
    dict(k_blocks_per_stage=4, stages=3, rows_per_stage=24),
    dict(k_blocks_per_stage=8, stages=2, rows_per_stage=64),
    dict(k_blocks_per_stage=4, stages=3, token_tile=32),
    dict(k_blocks_per_stage=4, stages=3, token_tile=48),
    dict(k_blocks_per_stage=4, stages=3, token_tile=64),
]


@pytest.mark.parametrize("cfg", SPLIT_CONFIGS, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
@pytest.mark.parametrize("M", [1, 13])
def test_split_configs(cfg, M):
    p = inputs.make_problem(M, 2056, 3592, seed=31 + M)
    compare(run_split(p, **cfg), oracle_full(p.A, p.W, p.R), f"split M={M} {cfg}")


def test_split_deterministic_with_and_without_pdl():
    """Both halves' partial sums are added in one fixed order: repeated runs,
    with and without programmatic dependent launch, give the same bits."""
    p = inputs.make_problem(12, N_DOWN, K_DOWN, seed=77)
    y1 = run_split(p)
    y2 = run_split(p)
    y3 = run_split(p, flags=sgr.SGR_FLAG_NO_PDL)
    assert np.array_equal(y1, y2) and np.array_equal(y1, y3)


def test_split_strided_and_in_place():
    M, N, K = 10, 2048, 3584
    p = inputs.make_problem(M, N, K, seed=59)
    Abig = torch.zeros((M, K + 128), dtype=torch.bfloat16, device="cuda")
    A = Abig[:, 64:64 + K]
    A.copy_(p.A)
    big = torch.full((M, N + 256), 3.0, dtype=torch.bfloat16, device="cuda")
    RY = big[:, 128:128 + N]
    RY.copy_(p.R)
    sgr.skinny_gemm_residual_ex(A, p.W.cuda(), RY, RY, config=sgr.make_config(path=ROWS, k_split=2))
    torch.cuda.synchronize()
    compare(bits(RY), oracle_full(p.A, p.W, p.R), "split strided in-place")
    assert torch.all(big[:, :128] == 3.0) and torch.all(big[:, 128 + N:] == 3.0)


def test_split_integer_inputs_exact():
    M, N, K = 16, 1024, 4096
    A = inputs.integer_bf16((M, K), -2, 2, 34)
    W = inputs.integer_bf16((N, K), -2, 2, 35)
    R = inputs.integer_bf16((M, N), -8, 8, 36)
    want = A.to(torch.int64) @ W.to(torch.int64).T + R.to(torch.int64)
    assert want.abs().max() < 2 ** 24
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    sgr.skinny_gemm_residual_ex(A.cuda(), W.cuda(), R.cuda(), Y, config=sgr.make_config(path=ROWS, k_split=2))
    torch.cuda.synchronize()
    assert torch.equal(Y.cpu(), want.to(torch.bfloat16))


def test_split_pdl_chain_in_graph_matches_oracle():
    """Three dependent split calls in one CUDA graph (A_i = Y_{i-1}[:, :K]),
    launched with programmatic dependent launch."""
    M, N, K = 8, 2048, 2048
    Ws = [inputs.make_weights(N, K, seed=700 + i) for i in range(3)]
    Rs = [inputs.make_rows(M, N, seed=710 + i) for i in range(3)]
    A0 = inputs.make_rows(M, K, seed=720)
    dW, dR, dA0 = [w.cuda() for w in Ws], [r.cuda() for r in Rs], A0.cuda()
    Ys = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    cfg = sgr.make_config(path=ROWS, k_split=2)
    stream = torch.cuda.Stream()

    def run():
        for i in range(3):
            A = dA0 if i == 0 else Ys[i - 1][:, :K]
            sgr.skinny_gemm_residual_ex(A, dW[i], dR[i], Ys[i], config=cfg, stream=stream)

    with torch.cuda.stream(stream):
        run()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        run()
    for Y in Ys:
        Y.fill_(float("nan"))
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    A = A0
    for i in range(3):
        compare(bits(Ys[i]), oracle_full(A, Ws[i], Rs[i]), f"split chain layer {i}")
        A = Ys[i].cpu()[:, :K]


def test_split_rejects_unsupported_forms():
    p = inputs.make_problem(20, 2048, 1024, seed=1)
    A, W, R = (t.cuda() for t in (p.A, p.W, p.R))
    for cfg in (dict(k_split=3), dict(k_split=-1), dict(k_split=2, token_tile=128),
                dict(k_split=2, token_tile=80), dict(k_split=2, rows_per_stage=20)):
        with pytest.raises(sgr.SgrError) as e:
            sgr.skinny_gemm_residual_ex(A, W, R, config=sgr.make_config(path=ROWS, **cfg))
        assert e.value.status == sgr.SGR_ERR_UNSUPPORTED, cfg
    q = inputs.make_problem(4, 2048, 1024, seed=2)
    with pytest.raises(sgr.SgrError) as e:  # the grouped kernel's 64-token tile has no split form
        sgr.skinny_gemm_residual_grouped([(q.A.cuda(), q.W.cuda(), q.R.cuda(), None)],
                                         config=sgr.make_config(path=ROWS, k_split=2, token_tile=64))
    assert e.value.status == sgr.SGR_ERR_UNSUPPORTED


@pytest.mark.parametrize("nt,kb,st,counts", [(16, 8, 3, [1, 5, 0, 16]), (48, 4, 4, [33, 2, 48])])
def test_split_grouped_matches_oracle_and_separate_calls(nt, kb, st, counts):
    """The grouped launch with the K split (a cluster per slab and problem):
    every element against the oracle, and the same bits as separate calls
    with the same configuration."""
    probs = [inputs.make_problem(m, N_DOWN, K_DOWN, seed=900 + 13 * i + m) for i, m in enumerate(counts)]
    dev = [(p.A.cuda(), p.W.cuda(), p.R.cuda(), None) for p in probs]
    cfg = sgr.make_config(path=ROWS, k_split=2, token_tile=nt, k_blocks_per_stage=kb, stages=st)
    ys = sgr.skinny_gemm_residual_grouped(dev, config=cfg)
    torch.cuda.synchronize()
    for i, (p, y) in enumerate(zip(probs, ys)):
        if p.A.shape[0] == 0:
            continue
        compare(bits(y), oracle_full(p.A, p.W, p.R), f"grouped split expert {i} M={p.A.shape[0]}")
        sep = sgr.skinny_gemm_residual_ex(dev[i][0], dev[i][1], dev[i][2], config=cfg)
        torch.cuda.synchronize()
        assert np.array_equal(bits(sep), bits(y)), i


# Untabulated shapes whose default configuration takes the split (slabs of at
# most 32 rows over K >= 4096), through the library's own choice.
AUTO_SPLIT = [(1, 2048, 8192), (16, 2048, 8192), (40, 2560, 10240), (64, 1024, 4096), (7, 4096, 14336),
              (33, 1000, 4104)]


@pytest.mark.parametrize("M,N,K", AUTO_SPLIT)
def test_split_default_configuration_every_element(M, N, K):
    c = sgr.sgr_default_config(M, N, K)
    assert (c.path, c.k_split) == (ROWS, 2), (c.path, c.k_split)
    p = inputs.make_problem(M, N, K, seed=800 + M + N)
    Y = sgr.skinny_gemm_residual(p.A.cuda(), p.W.cuda(), p.R.cuda())
    torch.cuda.synchronize()
    compare(bits(Y), oracle_full(p.A, p.W, p.R), f"split default {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K,split", [(16, 7168, 3584, 0), (16, 3584, 7168, 2), (64, 3584, 7168, 2),
                                         (16, 7168, 2048, 0), (16, 2048, 2048, 0)])
def test_split_default_choice(M, N, K, split):
    """The measured table (up- and down-projection) and the default rule for
    other shapes: 48-row slabs and short K stay unsplit."""
    c = sgr.sgr_default_config(M, N, K)
    assert (c.k_split == 2) == (split == 2), (M, N, K, c.path, c.k_split)

