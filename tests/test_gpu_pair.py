"""GPU parity of the 2-CTA tile GEMM (tcgen05 cta_group::2: 256-token x
tile_n tiles computed by a CTA pair, each CTA loading its own tokens and half
of the W tile) against the CPU oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import skinny_bf16_gemm_residual_gb300 as sgr
from skinny_bf16_gemm_residual_gb300 import inputs
from parity import bits, compare, oracle_full, oracle_problem

pytestmark = pytest.mark.gpu

N_FULL, K_FULL = inputs.N_LATENT_MOE, inputs.K_LATENT_MOE
PAIR = sgr.SGR_PATH_PAIR


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    torch.cuda.set_device(0)
    sgr.sgr_init(0)
    sgr.sgr_device_error(0, clear=True)
    yield
    assert sgr.sgr_device_error(0) == 0, "a kernel reported a timed-out wait"


def run_pair(p, **cfg):
    A, W, R = (t.cuda() for t in (p.A, p.W, p.R))
    Y = torch.full_like(R, float("nan"))
    sgr.skinny_gemm_residual_ex(A, W, R, Y, config=sgr.make_config(path=PAIR, **cfg))
    torch.cuda.synchronize()
    return bits(Y)


def test_pair_tiny():
    """One pair, one tile, two K blocks: the smallest case of the kernel."""
    p = inputs.make_problem(256, 64, 128, seed=1)
    compare(run_pair(p, tile_n=64), oracle_full(p.A, p.W, p.R), "pair tiny")


# Ragged in every dimension: M below, at and across the 256-token tile and
# its 128-token halves; N not a multiple of the tile width; K not a multiple
# of the 64-wide K block, and a single partial block.
SMALL = [(1, 520, 264), (5, 304, 8), (100, 1024, 520), (128, 256, 64), (129, 392, 1000), (255, 264, 1000),
         (256, 256, 128), (257, 1000, 136), (383, 1000, 136), (512, 2056, 1800), (640, 776, 3584)]


@pytest.mark.parametrize("tile_n", [0, 64, 96, 128, 192, 256])
@pytest.mark.parametrize("M,N,K", SMALL)
def test_pair_small_shapes(M, N, K, tile_n):
    p = inputs.make_problem(M, N, K, seed=M * 7 + N + K)
    compare(run_pair(p, tile_n=tile_n), oracle_full(p.A, p.W, p.R), f"pair {M}x{N}x{K} nt={tile_n}")


@pytest.mark.parametrize("M", [256, 512, 1024, 1000])
def test_pair_full_size_compute_bound_every_element(M):
    """The compute-bound sweep at the latent-MoE shape: every element."""
    p, ref = oracle_problem(M, N_FULL, K_FULL, seed=M)
    m = compare(run_pair(p), ref, f"pair M={M}")
    assert m["cosine"] > 0.999


@pytest.mark.parametrize("M", [128, 384])
def test_pair_full_size_other_m(M):
    p = inputs.make_problem(M, N_FULL, K_FULL, seed=M + 3)
    compare(run_pair(p), oracle_full(p.A, p.W, p.R), f"pair M={M}")


PAIR_CONFIGS = [
    dict(tile_n=64, stages=2),
    dict(tile_n=96, k_blocks_per_stage=1, stages=10),
    dict(tile_n=128, stages=4, prefetch_stages=2),
    dict(tile_n=192, k_blocks_per_stage=1, stages=8),
    dict(tile_n=192, stages=3, prefetch_stages=1),
    dict(tile_n=256, k_blocks_per_stage=1, stages=7),
    dict(tile_n=256, stages=2),
    dict(tile_n=128, k_blocks_per_stage=2, stages=4),
    dict(tile_n=192, k_blocks_per_stage=2, stages=3),
    dict(tile_n=96, k_blocks_per_stage=4, stages=2, prefetch_stages=1),
]


@pytest.mark.parametrize("cfg", PAIR_CONFIGS, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
@pytest.mark.parametrize("M", [1, 300, 700])
def test_pair_configs(cfg, M):
    N, K = 2056, 1032
    p = inputs.make_problem(M, N, K, seed=23 + M)
    compare(run_pair(p, **cfg), oracle_full(p.A, p.W, p.R), f"pair M={M} {cfg}")


def test_pair_many_tiles_per_pair():
    """More tiles than pairs (several tiles per persistent pair, both
    accumulators in use, phase parities wrapping)."""
    M, N, K = 2048, 4096, 256
    p = inputs.make_problem(M, N, K, seed=77)
    compare(run_pair(p, tile_n=64), oracle_full(p.A, p.W, p.R), "pair many tiles")


def test_pair_strided_in_place_and_deterministic():
    M, N, K = 300, 1024, 1032
    p = inputs.make_problem(M, N, K, seed=58)
    cfg = dict(tile_n=128)
    Abig = torch.zeros((M, K + 136), dtype=torch.bfloat16, device="cuda")
    A = Abig[:, 64:64 + K]
    A.copy_(p.A)
    big = torch.full((M, N + 512), 3.0, dtype=torch.bfloat16, device="cuda")
    RY = big[:, 256:256 + N]
    RY.copy_(p.R)
    sgr.skinny_gemm_residual_ex(A, p.W.cuda(), RY, RY, config=sgr.make_config(path=PAIR, **cfg))
    torch.cuda.synchronize()
    compare(bits(RY), oracle_full(p.A, p.W, p.R), "pair strided in-place")
    assert torch.all(big[:, :256] == 3.0) and torch.all(big[:, 256 + N:] == 3.0)
    y1, y2 = run_pair(p, **cfg), run_pair(p, **cfg)
    assert np.array_equal(y1, y2) and np.array_equal(y1, bits(RY))


def test_pair_integer_inputs_exact():
    M, N, K = 300, 1024, 1024
    A = inputs.integer_bf16((M, K), -2, 2, 24)
    W = inputs.integer_bf16((N, K), -2, 2, 25)
    R = inputs.integer_bf16((M, N), -8, 8, 26)
    want = A.to(torch.int64) @ W.to(torch.int64).T + R.to(torch.int64)
    assert want.abs().max() < 2 ** 24
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    sgr.skinny_gemm_residual_ex(A.cuda(), W.cuda(), R.cuda(), Y, config=sgr.make_config(path=PAIR))
    torch.cuda.synchronize()
    assert torch.equal(Y.cpu(), want.to(torch.bfloat16))


def test_pair_pdl_chain_matches_oracle():
    """Three dependent pair-kernel calls, each reading the previous output as
    its activations (A_i = Y_{i-1}[:, :K]), launched with programmatic
    dependent launch in one CUDA graph."""
    M, N, K = 512, 2048, 1024
    Ws = [inputs.make_weights(N, K, seed=300 + i) for i in range(3)]
    Rs = [inputs.make_rows(M, N, seed=310 + i) for i in range(3)]
    A0 = inputs.make_rows(M, K, seed=320)
    dW, dR = [w.cuda() for w in Ws], [r.cuda() for r in Rs]
    dA0 = A0.cuda()
    Ys = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    cfg = sgr.make_config(path=PAIR)
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
        ref = oracle_full(A, Ws[i], Rs[i])
        compare(bits(Ys[i]), ref, f"pair chain layer {i}")
        A = Ys[i].cpu()[:, :K]  # the GPU's output feeds the next layer, as in the chain


def test_pair_rejects_bad_config():
    p = inputs.make_problem(300, 256, 256, seed=1)
    A, W, R = (t.cuda() for t in (p.A, p.W, p.R))
    for cfg in (dict(tile_n=80), dict(tile_n=320), dict(tile_n=32), dict(ctas_per_sm=2), dict(tile_n=256, stages=8),
                dict(tile_n=64, stages=3, prefetch_stages=4), dict(stages=17), dict(token_tile=128),
                dict(k_blocks_per_stage=3), dict(k_split=2)):
        with pytest.raises(sgr.SgrError) as e:
            sgr.skinny_gemm_residual_ex(A, W, R, config=sgr.make_config(path=PAIR, **cfg))
        assert e.value.status == sgr.SGR_ERR_UNSUPPORTED, cfg


def test_pair_kernel_resources():
    r = sgr.sgr_kernel_resources(1024, N_FULL, K_FULL, path=PAIR)
    assert r["spill_bytes"] == 0 and r["threads"] == 192 and r["smem_bytes"] <= 232448, r
