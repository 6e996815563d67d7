"""The seeded input generators that the CUDA path's tests, the benchmark and
the oracle's checks share: same seed gives the same bits, the stated draw order
and distributions hold, and the FP8 problems are the per-row absmax
quantisation they claim to be (checked with torch's own E4M3 conversion)."""
import math

import pytest
import torch

from skinny_bf16_gemm_residual_gb300 import inputs


def same(a: torch.Tensor, b: torch.Tensor) -> bool:
    return a.dtype == b.dtype and a.shape == b.shape and torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def test_same_seed_same_bits_other_seed_other_bits():
    p, q, r = (inputs.make_problem(4, 64, 128, seed=s) for s in (3, 3, 4))
    assert same(p.A, q.A) and same(p.W, q.W) and same(p.R, q.R)
    assert not torch.equal(p.A, r.A) and not torch.equal(p.W, r.W) and not torch.equal(p.R, r.R)
    w1, w2 = inputs.make_problem_w8(4, 64, 128, seed=7), inputs.make_problem_w8(4, 64, 128, seed=7)
    assert same(w1.Wq, w2.Wq) and torch.equal(w1.scale, w2.scale)


def test_shapes_and_dtypes():
    p = inputs.make_problem(5, 24, 40, seed=0)
    assert (p.M, p.N, p.K) == (5, 24, 40)
    assert p.A.shape == (5, 40) and p.W.shape == (24, 40) and p.R.shape == (5, 24)
    assert {t.dtype for t in (p.A, p.W, p.R)} == {torch.bfloat16}
    q = inputs.make_problem_w8(5, 24, 40, seed=0)
    assert (q.M, q.N, q.K) == (5, 24, 40)
    assert q.Wq.dtype == torch.uint8 and q.Wq.shape == (24, 40) and q.Wq.is_contiguous()
    assert q.scale.dtype == torch.float32 and q.scale.shape == (24,)


def test_distributions():
    K = 3584
    p = inputs.make_problem(64, 512, K, seed=1)
    for t, sd in ((p.A, 1.0), (p.R, 1.0), (p.W, 1.0 / math.sqrt(K))):
        x = t.double()
        assert abs(x.mean().item()) < 0.02 * sd
        assert abs(x.std().item() / sd - 1.0) < 0.02


def test_fp8_problem_shares_the_bf16_draws():
    """Draw order A, W, R: the FP8 problem's A and R are the BF16 problem's, and
    its dequantised weights are the same W to E4M3 precision."""
    p, q = inputs.make_problem(3, 64, 256, seed=5), inputs.make_problem_w8(3, 64, 256, seed=5)
    assert same(p.A, q.A) and same(p.R, q.R)
    deq = q.Wq.view(torch.float8_e4m3fn).double() * q.scale.double()[:, None]
    W = p.W.double()
    # E4M3 keeps 3 fraction bits (relative error <= 2^-4 for normals); subnormal
    # codes are spaced scale * 2^-9; the BF16 W adds its own 2^-9 relative error.
    bound = W.abs() * (2.0 ** -4 + 2.0 ** -8) + q.scale.double()[:, None] * 2.0 ** -9
    assert bool(((deq - W).abs() <= bound).all())


def test_fp8_rows_use_the_full_code_range():
    q = inputs.make_problem_w8(2, 128, 512, seed=9)
    vals = q.Wq.view(torch.float8_e4m3fn).float()
    assert bool((vals.abs().amax(dim=1) == inputs.E4M3_MAX).all())  # every row's absmax maps to +-448
    assert not bool(((q.Wq & 0x7F) == 0x7F).any())                  # no NaN code
    assert bool((q.scale > 0).all()) and bool(torch.isfinite(q.scale).all())


def test_fp8_problem_edge_shapes():
    q = inputs.make_problem_w8(2, 8, 0, seed=0)  # empty K: unit scales, no codes
    assert q.Wq.shape == (8, 0) and bool((q.scale == 1).all())
    z = inputs.make_problem_w8(0, 16, 32, seed=0)
    assert z.A.shape == (0, 32) and z.R.shape == (0, 16) and z.Wq.shape == (16, 32)


def test_random_codes_cover_every_finite_pattern():
    c = inputs.random_e4m3_codes((64, 1024), seed=2)
    assert c.dtype == torch.uint8
    seen = set(torch.unique(c).tolist())
    assert seen == set(range(256)) - {0x7F, 0xFF}
    n = inputs.random_e4m3_codes((64, 1024), seed=2, nan=True)
    assert {0x7F, 0xFF} <= set(torch.unique(n).tolist())


@pytest.mark.parametrize("lo,hi", [(-12, 2), (-14, -8), (0, 0)])
def test_random_scales_range(lo, hi):
    s = inputs.random_scales(4096, seed=3, lo_exp=lo, hi_exp=hi)
    assert s.dtype == torch.float32
    e = torch.floor(torch.log2(s.double()))
    assert int(e.min()) >= lo and int(e.max()) <= hi
    assert int(e.min()) == lo and int(e.max()) == hi  # both ends drawn at this size


def test_wide_exponent_and_integer_generators_are_exact():
    b = inputs.random_bf16_bits((256, 64), seed=4, lo_exp=-12, hi_exp=6)
    x = b.double()
    e = torch.floor(torch.log2(x.abs()))
    assert int(e.min()) == -12 and int(e.max()) == 6
    assert torch.equal(x.to(torch.bfloat16).double(), x)
    i = inputs.integer_bf16((128, 64), -5, 9, seed=5).double()
    assert torch.equal(i, torch.round(i)) and int(i.min()) == -5 and int(i.max()) == 9


def _w4_dequantised(q) -> torch.Tensor:
    """e2m1(code) * e4m3(block scale) * gs from the fields (float64, [N, K])."""
    lo, hi = (q.Wq4 & 15).long(), (q.Wq4 >> 4).long()
    codes = torch.stack((lo, hi), dim=2).reshape(q.Wq4.shape[0], -1)
    mag = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=torch.float64)[codes & 7]
    val = torch.where(codes >= 8, -mag, mag)
    sc = q.bs.view(torch.float8_e4m3fn).double().repeat_interleave(16, dim=1)[:, :codes.shape[1]]
    return val * sc * q.gs


def test_nvfp4_problem_shares_the_bf16_draws():
    """Draw order A, W, R as in the BF16 problem; the dequantised NVFP4 weights
    are W to within half an E2M1 step of the block's scale (the largest step
    is 2, between 4 and 6) plus the E4M3 rounding of that scale."""
    p, q = inputs.make_problem(3, 64, 256, seed=5), inputs.make_problem_w4(3, 64, 256, seed=5)
    assert same(p.A, q.A) and same(p.R, q.R)
    deq = _w4_dequantised(q)
    W = p.W.double()
    blk = q.bs.view(torch.float8_e4m3fn).double().repeat_interleave(16, dim=1) * q.gs
    bound = blk * 1.0 + W.abs() * (2.0 ** -3 + 2.0 ** -8)
    assert bool(((deq - W).abs() <= bound).all())
    cos = float((deq * W).sum() / (deq.norm() * W.norm()))
    assert cos > 0.99


def test_nvfp4_problem_layout_and_range():
    q = inputs.make_problem_w4(2, 32, 512, seed=9)
    assert q.Wq4.dtype == torch.uint8 and q.Wq4.shape == (32, 256)
    assert q.bs.dtype == torch.uint8 and q.bs.shape == (32, 32)
    assert not bool(((q.bs & 0x7F) == 0x7F).any()) and not bool((q.bs >= 0x80).any())  # finite, positive scales
    assert q.gs > 0
    codes = torch.cat(((q.Wq4 & 15), (q.Wq4 >> 4)))
    assert len(set(torch.unique(codes).tolist())) >= 14  # both signs of every magnitude (up to +-0)
    with pytest.raises(ValueError):
        inputs.make_problem_w4(1, 8, 15, seed=0)  # odd K cannot be packed


def test_random_e2m1_bytes_cover_every_code_pair():
    b = inputs.random_e2m1_bytes((64, 256), seed=4)
    assert b.dtype == torch.uint8 and set(torch.unique(b).tolist()) == set(range(256))
