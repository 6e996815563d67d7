"""GPU parity of the grouped (mixture-of-experts) call: every group against
the CPU oracle, with synthetic routing (token counts per expert from a seeded
top-k assignment, including experts that receive no token)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import skinny_bf16_gemm_residual_gb300 as sgr
from skinny_bf16_gemm_residual_gb300 import inputs
from parity import bits, compare, oracle_full

pytestmark = pytest.mark.gpu

N_FULL, K_FULL = inputs.N_LATENT_MOE, inputs.K_LATENT_MOE


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    torch.cuda.set_device(0)
    sgr.sgr_init(0)
    sgr.sgr_device_error(0, clear=True)
    yield
    assert sgr.sgr_device_error(0) == 0, "a kernel reported a timed-out wait"


def expert_problems(counts, N, K, seed):
    return [inputs.make_problem(m, N, K, seed=seed + 17 * e) for e, m in enumerate(counts)]


def check(counts, N, K, seed, **kw):
    probs = expert_problems(counts, N, K, seed)
    dev = [(p.A.cuda(), p.W.cuda(), p.R.cuda(), None) for p in probs]
    ys = sgr.skinny_gemm_residual_grouped(dev, **kw)
    torch.cuda.synchronize()
    for e, (p, y) in enumerate(zip(probs, ys)):
        if p.A.shape[0]:
            compare(bits(y), oracle_full(p.A, p.W, p.R), f"expert {e} M={p.A.shape[0]}")


@pytest.mark.parametrize("counts", [[4], [1, 2, 3, 16], [0, 5, 0, 16, 1], [8] * 8, [16, 0, 0, 0]])
def test_grouped_full_size(counts):
    check(counts, N_FULL, K_FULL, seed=sum(counts))


@pytest.mark.parametrize("N,K", [(1000, 264), (304, 8), (3584, 7168), (2056, 1800), (2048, 8192)])
def test_grouped_small_and_other_shapes(N, K):
    check([3, 0, 16, 1, 7], N, K, seed=N + K)


def test_grouped_synthetic_top2_routing():
    """16 tokens routed top-2 over 8 experts: per-expert counts from a seeded draw."""
    rng = np.random.default_rng(7)
    choice = np.stack([rng.choice(8, size=2, replace=False) for _ in range(16)])
    counts = np.bincount(choice.ravel(), minlength=8).tolist()
    check(counts, N_FULL, K_FULL, seed=99)


def test_grouped_more_than_32_experts_and_larger_batches():
    counts = [(e * 5) % 19 for e in range(40)]  # 40 experts -> two launches; up to 18 tokens
    check(counts, 1024, 520, seed=5)
    check([40, 0, 100, 256], 2056, 1032, seed=6)


def test_grouped_in_place_and_strided():
    p = inputs.make_problem(6, 2056, 1032, seed=11)
    q = inputs.make_problem(3, 2056, 1032, seed=12)
    big = torch.zeros((6, 2056 + 256), dtype=torch.bfloat16, device="cuda")
    ry = big[:, 128:128 + 2056]
    ry.copy_(p.R)
    y2 = torch.empty((3, 2056), dtype=torch.bfloat16, device="cuda")
    sgr.skinny_gemm_residual_grouped([(p.A.cuda(), p.W.cuda(), ry, ry), (q.A.cuda(), q.W.cuda(), q.R.cuda(), y2)])
    torch.cuda.synchronize()
    compare(bits(ry), oracle_full(p.A, p.W, p.R), "in place")
    compare(bits(y2), oracle_full(q.A, q.W, q.R), "second expert")
    assert torch.all(big[:, :128] == 0) and torch.all(big[:, 128 + 2056:] == 0)


def test_grouped_matches_separate_calls_bitwise():
    counts = [2, 9, 16]
    probs = expert_problems(counts, N_FULL, K_FULL, seed=21)
    dev = [(p.A.cuda(), p.W.cuda(), p.R.cuda(), None) for p in probs]
    cfg = sgr.make_config(path=sgr.SGR_PATH_TC_ROWS, k_blocks_per_stage=8, stages=3, token_tile=16)
    ys = sgr.skinny_gemm_residual_grouped(dev, config=cfg)
    sep = [sgr.skinny_gemm_residual_ex(A, W, R, config=cfg) for A, W, R, _ in dev]
    torch.cuda.synchronize()
    for a, b in zip(ys, sep):
        assert np.array_equal(bits(a), bits(b))


def test_grouped_rejects_other_paths():
    p = inputs.make_problem(4, 256, 256, seed=1)
    with pytest.raises(sgr.SgrError) as e:
        sgr.skinny_gemm_residual_grouped([(p.A.cuda(), p.W.cuda(), p.R.cuda(), None)],
                                         config=sgr.make_config(path=sgr.SGR_PATH_TILE))
    assert e.value.status == sgr.SGR_ERR_UNSUPPORTED
