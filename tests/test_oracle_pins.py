"""The CPU oracle against its pins (no GPU)."""
import numpy as np
import pytest

import pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(oracle_lib, check):
    check(oracle_lib)


def test_oracle_threads_do_not_change_bits(oracle_lib):
    from skinny_bf16_gemm_residual_gb300 import inputs

    p = inputs.make_problem(3, N=257, K=96, seed=7)
    y1 = oracle_lib.gemm_residual(p.A, p.W, p.R, threads=1)
    y8 = oracle_lib.gemm_residual(p.A, p.W, p.R, threads=8)
    assert np.array_equal(y1, y8)


def test_oracle_sample_matches_full(oracle_lib):
    from skinny_bf16_gemm_residual_gb300 import inputs

    p = inputs.make_problem(4, N=300, K=128, seed=8)
    full = oracle_lib.gemm_residual(p.A, p.W, p.R)
    rng = np.random.default_rng(0)
    ms = rng.integers(0, 4, 50)
    ns = rng.integers(0, 300, 50)
    assert np.array_equal(oracle_lib.sample(p.A, p.W, p.R, ms, ns), full[ms, ns])


def test_oracle_unrounded_is_close_to_rounded(oracle_lib):
    """The rounded output is within half a BF16 ulp of the FP64 value."""
    from skinny_bf16_gemm_residual_gb300 import inputs

    p = inputs.make_problem(2, N=64, K=256, seed=9)
    t = oracle_lib.gemm_residual_f64(p.A, p.W, p.R)
    y = oracle_lib.gemm_residual(p.A, p.W, p.R)
    yv = (y.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ulp = 2.0 ** (np.floor(np.log2(np.abs(t))) - 7)
    assert np.all(np.abs(yv - t) <= ulp / 2)


def test_oracle_empty_shapes(oracle_lib):
    A = np.zeros((0, 8), np.uint16)
    W = np.zeros((4, 8), np.uint16)
    R = np.zeros((0, 4), np.uint16)
    assert oracle_lib.gemm_residual(A, W, R).shape == (0, 4)
    # K = 0: the product is an empty sum, Y = R
    A0 = np.zeros((2, 0), np.uint16)
    W0 = np.zeros((3, 0), np.uint16)
    R0 = np.full((2, 3), 0x3F80, np.uint16)
    assert np.array_equal(oracle_lib.gemm_residual(A0, W0, R0), R0)
