"""Seeded random shapes, strides and paths against the oracle: every case is a
fresh (M, N, K) with N, K multiples of 8, row strides padded at random, Y
either a separate buffer or the residual itself (in place), on the library's
own path choice or a forced one.  Sizes stay small enough for the oracle to
check every element."""
import numpy as np
import pytest
import torch

import skinny_bf16_gemm_residual_gb300 as sgr
from skinny_bf16_gemm_residual_gb300 import inputs
from parity import bits, compare, oracle_full

import oracle

pytestmark = pytest.mark.gpu

PATHS = [sgr.SGR_PATH_AUTO, sgr.SGR_PATH_TC_ROWS, sgr.SGR_PATH_TILE, sgr.SGR_PATH_TC, sgr.SGR_PATH_SIMT]


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    torch.cuda.set_device(0)
    sgr.sgr_init(0)
    sgr.sgr_device_error(0, clear=True)
    yield
    assert sgr.sgr_device_error(0) == 0, "a kernel reported a timed-out wait"


def padded(t: torch.Tensor, pad: int) -> torch.Tensor:
    """A CUDA copy of `t` whose rows sit in a wider buffer (row stride + pad)."""
    rows, cols = t.shape
    buf = torch.zeros((rows, cols + pad), dtype=t.dtype, device="cuda")
    view = buf[:, pad // 2 // 8 * 8:pad // 2 // 8 * 8 + cols]
    view.copy_(t)
    return view


def case(seed: int):
    rng = np.random.default_rng(seed)
    M = int(rng.choice([1, 2, 3, 5, 8, 13, 16, 24, 40, 64, 100, 128, 200, 256]))
    N = int(rng.integers(1, 96)) * 8
    K = int(rng.integers(1, 80)) * 8
    return rng, M, N, K


@pytest.mark.parametrize("seed", range(40))
def test_fuzz_bf16(seed):
    rng, M, N, K = case(seed)
    path = PATHS[seed % len(PATHS)]
    if path == sgr.SGR_PATH_SIMT and M > 16:
        path = sgr.SGR_PATH_AUTO
    p = inputs.make_problem(M, N, K, seed=1000 + seed)
    A = padded(p.A, int(rng.integers(0, 4)) * 8)
    R = padded(p.R, int(rng.integers(0, 4)) * 8)
    in_place = bool(rng.integers(0, 2))
    Y = R if in_place else padded(torch.zeros_like(p.R), int(rng.integers(0, 4)) * 8)
    cfg = None if path == sgr.SGR_PATH_AUTO else sgr.make_config(path=path)
    try:
        sgr.skinny_gemm_residual_ex(A, p.W.cuda(), R, Y, config=cfg)
    except sgr.SgrError as e:  # a forced path may not hold the shape; the library's choice must
        assert path != sgr.SGR_PATH_AUTO and e.status == sgr.SGR_ERR_UNSUPPORTED, (M, N, K, path, e)
        return
    torch.cuda.synchronize()
    compare(bits(Y), oracle_full(p.A, p.W, p.R), f"fuzz bf16 seed={seed} M={M} N={N} K={K} path={path}")


@pytest.mark.parametrize("seed", range(24))
def test_fuzz_rows_ksplit(seed):
    """The row slab with the 2-CTA K split on seeded random shapes (1-64
    tokens, K up to 8 192), ring shapes, row strides and in-place outputs."""
    rng = np.random.default_rng(5000 + seed)
    M = int(rng.integers(1, 65))
    N = int(rng.integers(1, 600)) * 8
    K = int(rng.integers(1, 1025)) * 8
    kb = int(rng.choice([1, 2, 4, 8]))
    st = int(rng.integers(2, 7))
    p = inputs.make_problem(M, N, K, seed=6000 + seed)
    A = padded(p.A, int(rng.integers(0, 4)) * 8)
    R = padded(p.R, int(rng.integers(0, 4)) * 8)
    in_place = bool(rng.integers(0, 2))
    Y = R if in_place else padded(torch.zeros_like(p.R), int(rng.integers(0, 4)) * 8)
    cfg = sgr.make_config(path=sgr.SGR_PATH_TC_ROWS, k_split=2, k_blocks_per_stage=kb, stages=st)
    try:
        sgr.skinny_gemm_residual_ex(A, p.W.cuda(), R, Y, config=cfg)
    except sgr.SgrError as e:  # a ring too large for shared memory, or too small for the hand-over
        assert e.status == sgr.SGR_ERR_UNSUPPORTED, (M, N, K, kb, st, e)
        return
    torch.cuda.synchronize()
    compare(bits(Y), oracle_full(p.A, p.W, p.R), f"fuzz k-split seed={seed} M={M} N={N} K={K} kb={kb} st={st}")


@pytest.mark.parametrize("seed", range(32))
def test_fuzz_w8(seed):
    rng, M, N, K = case(500 + seed)
    K = (K + 15) // 16 * 16 if seed % 2 else K  # half the cases have K a multiple of 16
    path = (sgr.SGR_PATH_AUTO, sgr.SGR_PATH_W8, sgr.SGR_PATH_SIMT, sgr.SGR_PATH_W8S)[seed % 4]
    p = inputs.make_problem_w8(M, N, K, seed=2000 + seed)
    if seed % 4 == 0:  # codes of every kind and random scales
        p = inputs.ProblemW8(p.A, inputs.random_e4m3_codes((N, K), 3000 + seed),
                             inputs.random_scales(N, 4000 + seed, lo_exp=-14, hi_exp=-8), p.R, p.seed)
    pad = 16 * int(rng.integers(0, 3)) + ((-K) % 16)
    Wbuf = torch.zeros((N, K + pad), dtype=torch.uint8, device="cuda")
    Wq = Wbuf[:, :K]
    Wq.copy_(p.Wq)
    A = padded(p.A, int(rng.integers(0, 4)) * 8)
    R = padded(p.R, int(rng.integers(0, 4)) * 8)
    Y = R if bool(rng.integers(0, 2)) else None
    cfg = None if path == sgr.SGR_PATH_AUTO else sgr.make_config(path=path)
    try:
        Y = sgr.skinny_gemm_residual_w8(A, Wq, p.scale.cuda(), R, Y, config=cfg)
    except sgr.SgrError as e:
        assert path != sgr.SGR_PATH_AUTO and e.status == sgr.SGR_ERR_UNSUPPORTED, (M, N, K, path, e)
        return
    torch.cuda.synchronize()
    want = oracle.load().gemm_residual_w8(p.A, p.Wq, p.scale, p.R)
    compare(bits(Y), want, f"fuzz w8 seed={seed} M={M} N={N} K={K} path={path}")


@pytest.mark.parametrize("seed", range(32))
def test_fuzz_w4(seed):
    """NVFP4 weights: random shapes (K a multiple of 32 in half the cases),
    padded code and scale rows, random codes and block scales in a quarter
    of the cases, in place or not, on the library's choice or a forced kernel."""
    rng, M, N, K = case(700 + seed)
    K = (K + 31) // 32 * 32 if seed % 2 else K
    path = (sgr.SGR_PATH_AUTO, sgr.SGR_PATH_W8, sgr.SGR_PATH_SIMT)[seed % 3]
    p = inputs.make_problem_w4(M, N, K, seed=5000 + seed)
    if seed % 4 == 0:  # every code pair, random positive block scales, a random tensor scale
        bs = inputs.random_e4m3_codes((N, (K + 15) // 16), 6000 + seed) & 0x7F
        bs = torch.where(bs == 0x7F, bs - 1, bs)
        p = inputs.ProblemW4(p.A, inputs.random_e2m1_bytes((N, K // 2), 7000 + seed), bs,
                             float(inputs.random_scales(1, 8000 + seed, lo_exp=-8, hi_exp=-4)[0]), p.R, p.seed)
    half, nb = K // 2, (K + 15) // 16
    wpad = 16 * int(rng.integers(0, 3)) + ((-half) % 16)
    Wbuf = torch.zeros((N, half + wpad), dtype=torch.uint8, device="cuda")
    Wq4 = Wbuf[:, :half]
    Wq4.copy_(p.Wq4)
    spad = 16 * int(rng.integers(0, 3)) + ((-nb) % 16)
    Sbuf = torch.zeros((N, nb + spad), dtype=torch.uint8, device="cuda")
    bs = Sbuf[:, :nb]
    bs.copy_(p.bs)
    A = padded(p.A, int(rng.integers(0, 4)) * 8)
    R = padded(p.R, int(rng.integers(0, 4)) * 8)
    Y = R if bool(rng.integers(0, 2)) else None
    cfg = None if path == sgr.SGR_PATH_AUTO else sgr.make_config(path=path)
    try:
        Y = sgr.skinny_gemm_residual_w4(A, Wq4, bs, p.gs, R, Y, config=cfg)
    except sgr.SgrError as e:
        assert path != sgr.SGR_PATH_AUTO and e.status == sgr.SGR_ERR_UNSUPPORTED, (M, N, K, path, e)
        return
    torch.cuda.synchronize()
    want = oracle.load().gemm_residual_w4(p.A, p.Wq4, p.bs, p.gs, p.R)
    compare(bits(Y), want, f"fuzz w4 seed={seed} M={M} N={N} K={K} path={path}")

