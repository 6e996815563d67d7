"""Seeded synthetic inputs for the skinny BF16 projection GEMM + residual.

This module only draws random numbers; it holds none of the operation's
arithmetic, so both the CUDA path's tests/benchmark and the CPU oracle's
checks can take their inputs from it.

Shapes and distributions follow the decode-sized latent-MoE projection of the
vLLM "benchmark_k3_cutedsl_residual.py" page (module docstring and the N / K
constants: BF16[M,3584] @ BF16[7168,3584].T + BF16[M,7168]).  That page draws
every operand from a unit normal on the device; here W is scaled by 1/sqrt(K)
so that A.W^T has unit variance like R, which keeps Y ~ N(0, 2) and makes the
BF16 rounding of the output a relative 2^-9 effect.  Values are drawn on the
host (torch CPU generator, one per seed) in the order A, W, R and then copied
wherever they are needed, so every consumer sees the same bits.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

N_LATENT_MOE = 7168
K_LATENT_MOE = 3584


@dataclass
class Problem:
    """One synthetic problem: A [M,K], W [N,K], R [M,N], all torch.bfloat16 (CPU)."""

    A: torch.Tensor
    W: torch.Tensor
    R: torch.Tensor
    seed: int

    @property
    def M(self) -> int:
        return self.A.shape[0]

    @property
    def N(self) -> int:
        return self.W.shape[0]

    @property
    def K(self) -> int:
        return self.A.shape[1]


def make_problem(M: int, N: int = N_LATENT_MOE, K: int = K_LATENT_MOE, seed: int = 0,
                 w_scale: float | None = None) -> Problem:
    """A ~ N(0,1), W ~ N(0,1) * w_scale (default 1/sqrt(K)), R ~ N(0,1), BF16.

    Draw order A, W, R from ``torch.Generator().manual_seed(seed)``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    if w_scale is None:
        w_scale = 1.0 / math.sqrt(K) if K > 0 else 1.0
    A = torch.randn((M, K), generator=g, dtype=torch.float32).to(torch.bfloat16)
    W = (torch.randn((N, K), generator=g, dtype=torch.float32) * w_scale).to(torch.bfloat16)
    R = torch.randn((M, N), generator=g, dtype=torch.float32).to(torch.bfloat16)
    return Problem(A, W, R, seed)


def make_weights(N: int, K: int, seed: int, w_scale: float | None = None) -> torch.Tensor:
    """One W [N,K] BF16 ~ N(0,1)/sqrt(K) from its own seed (CPU)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    if w_scale is None:
        w_scale = 1.0 / math.sqrt(K) if K > 0 else 1.0
    return (torch.randn((N, K), generator=g, dtype=torch.float32) * w_scale).to(torch.bfloat16)


def make_rows(M: int, cols: int, seed: int) -> torch.Tensor:
    """[M, cols] BF16 ~ N(0,1) from its own seed (CPU): activations or residuals."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return torch.randn((M, cols), generator=g, dtype=torch.float32).to(torch.bfloat16)


def random_bf16_bits(shape, seed: int, lo_exp: int = -12, hi_exp: int = 6) -> torch.Tensor:
    """BF16 values with random sign, a random exponent in [lo_exp, hi_exp] and a
    random 7-bit fraction (CPU).  A wide exponent spread makes rounding matter."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    sign = torch.randint(0, 2, shape, generator=g) * 2 - 1
    expo = torch.randint(lo_exp, hi_exp + 1, shape, generator=g).to(torch.float64)
    frac = torch.randint(0, 128, shape, generator=g).to(torch.float64)
    vals = sign * (1.0 + frac / 128.0) * torch.pow(2.0, expo)
    return vals.to(torch.bfloat16)  # exactly representable: 8 significant bits


def integer_bf16(shape, lo: int, hi: int, seed: int) -> torch.Tensor:
    """Integer values in [lo, hi] stored as BF16 (exact for |v| <= 256) (CPU)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return torch.randint(lo, hi + 1, shape, generator=g).to(torch.bfloat16)


@dataclass
class ProblemW8:
    """A low-bit weight problem: A [M,K] BF16, Wq [N,K] FP8 E4M3 codes (torch.uint8),
    scale [N] float32 (one per output column), R [M,N] BF16 (all CPU)."""

    A: torch.Tensor
    Wq: torch.Tensor
    scale: torch.Tensor
    R: torch.Tensor
    seed: int

    @property
    def M(self) -> int:
        return self.A.shape[0]

    @property
    def N(self) -> int:
        return self.Wq.shape[0]

    @property
    def K(self) -> int:
        return self.A.shape[1]


E4M3_MAX = 448.0


def make_problem_w8(M: int, N: int = N_LATENT_MOE, K: int = K_LATENT_MOE, seed: int = 0) -> ProblemW8:
    """A, R ~ N(0,1) BF16 and per-column FP8 weights of a W ~ N(0,1)/sqrt(K).

    Draw order A, W, R from ``torch.Generator().manual_seed(seed)`` (the same
    draws as ``make_problem``).  Each row n of the float32 W gets the scale
    max|W[n,:]| / 448 (1 for an all-zero row) and the codes are torch's
    float32 -> float8_e4m3fn cast of W[n,:] / scale[n] (nearest, saturating):
    the per-channel absmax weight quantisation that produces such operands."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    A = torch.randn((M, K), generator=g, dtype=torch.float32).to(torch.bfloat16)
    W = torch.randn((N, K), generator=g, dtype=torch.float32) * (1.0 / math.sqrt(K) if K > 0 else 1.0)
    R = torch.randn((M, N), generator=g, dtype=torch.float32).to(torch.bfloat16)
    amax = W.abs().amax(dim=1) if K > 0 else torch.zeros(N)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax)).to(torch.float32)
    Wq = (W / scale[:, None]).to(torch.float8_e4m3fn).view(torch.uint8)
    return ProblemW8(A, Wq.contiguous(), scale.contiguous(), R, seed)


def random_e4m3_codes(shape, seed: int, nan: bool = False) -> torch.Tensor:
    """Uniformly random FP8 E4M3 codes (torch.uint8, CPU): every sign, exponent
    (subnormals and zero included) and fraction; the two NaN codes 0x7F / 0xFF
    only when ``nan``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    c = torch.randint(0, 256, shape, generator=g, dtype=torch.int64)
    if not nan:
        c = torch.where((c & 0x7F) == 0x7F, c - 1, c)
    return c.to(torch.uint8)


def random_scales(n: int, seed: int, lo_exp: int = -12, hi_exp: int = 2) -> torch.Tensor:
    """Positive float32 scales with random exponents in [lo_exp, hi_exp] and a
    random 23-bit fraction (CPU)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    expo = torch.randint(lo_exp, hi_exp + 1, (n,), generator=g).to(torch.float64)
    frac = torch.randint(0, 1 << 23, (n,), generator=g).to(torch.float64)
    return ((1.0 + frac / float(1 << 23)) * torch.pow(2.0, expo)).to(torch.float32)


@dataclass
class ProblemW4:
    """An NVFP4 weight problem: A [M,K] BF16; Wq4 [N,K/2] bytes (torch.uint8),
    each holding two E2M1 codes (element 2i in the low nibble); bs
    [N,ceil(K/16)] E4M3 block scales (torch.uint8); gs the tensor's float32
    scale; R [M,N] BF16 (all CPU)."""

    A: torch.Tensor
    Wq4: torch.Tensor
    bs: torch.Tensor
    gs: float
    R: torch.Tensor
    seed: int

    @property
    def M(self) -> int:
        return self.A.shape[0]

    @property
    def N(self) -> int:
        return self.Wq4.shape[0]

    @property
    def K(self) -> int:
        return self.A.shape[1]


E2M1_MAX = 6.0
_E2M1_LEVELS = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=torch.float32)
_E2M1_MIDPOINTS = (_E2M1_LEVELS[1:] + _E2M1_LEVELS[:-1]) / 2


def make_problem_w4(M: int, N: int = N_LATENT_MOE, K: int = K_LATENT_MOE, seed: int = 0) -> ProblemW4:
    """A, R ~ N(0,1) BF16 and NVFP4 weights of a W ~ N(0,1)/sqrt(K) (K even).

    Draw order A, W, R as in ``make_problem``.  Quantisation of the float32 W
    in blocks of 16 consecutive elements of a row: gs = max|W| / (6 * 448)
    (1 for an all-zero W); each block's scale is torch's float32 ->
    float8_e4m3fn cast of max|block| / (6 gs); each element's code is the
    E2M1 value nearest to w / (scale gs) (the lower one on a tie), with the
    sign of w: the NVFP4 weight quantisation that produces such operands."""
    if K % 2:
        raise ValueError("K must be even for packed 4-bit codes")
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    A = torch.randn((M, K), generator=g, dtype=torch.float32).to(torch.bfloat16)
    W = torch.randn((N, K), generator=g, dtype=torch.float32) * (1.0 / math.sqrt(K) if K > 0 else 1.0)
    R = torch.randn((M, N), generator=g, dtype=torch.float32).to(torch.bfloat16)
    nb = (K + 15) // 16
    Wp = torch.zeros((N, nb * 16), dtype=torch.float32)
    Wp[:, :K] = W
    amax = Wp.abs().reshape(N, nb, 16).amax(dim=2)
    top = float(amax.max()) if amax.numel() else 0.0
    gs = float(torch.tensor(top / (E2M1_MAX * E4M3_MAX) if top > 0 else 1.0, dtype=torch.float32))
    bs = (amax / (E2M1_MAX * gs)).to(torch.float8_e4m3fn)
    sval = bs.to(torch.float32).repeat_interleave(16, dim=1)[:, :K] * gs
    x = torch.where(sval > 0, W / torch.where(sval > 0, sval, torch.ones_like(sval)), torch.zeros_like(W))
    # Nearest level: the number of level midpoints strictly below |x| (the
    # lower level on a tie).
    idx = torch.searchsorted(_E2M1_MIDPOINTS, x.abs().contiguous(), right=False)
    codes = (idx | torch.where(x < 0, 8, 0)).to(torch.uint8)
    Wq4 = (codes[:, 0::2] | (codes[:, 1::2] << 4)).to(torch.uint8)
    return ProblemW4(A, Wq4.contiguous(), bs.view(torch.uint8).contiguous(), gs, R, seed)


def random_e2m1_bytes(shape, seed: int) -> torch.Tensor:
    """Uniformly random bytes (torch.uint8, CPU): two random E2M1 codes each,
    every sign, exponent and fraction (zero, the subnormal 0.5 and -0 included)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return torch.randint(0, 256, shape, generator=g, dtype=torch.int64).to(torch.uint8)

