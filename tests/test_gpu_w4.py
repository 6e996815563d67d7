"""GPU parity of the NVFP4-weight kernel (skinny_gemm_residual_w4: E2M1 codes,
E4M3 block scales per 16 elements, FP32 tensor scale) against the CPU
oracle's NVFP4 variant, element by element on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import skinny_bf16_gemm_residual_gb300 as sgr
from skinny_bf16_gemm_residual_gb300 import inputs
from parity import bits, compare

import oracle

pytestmark = pytest.mark.gpu

N_FULL, K_FULL = inputs.N_LATENT_MOE, inputs.K_LATENT_MOE
SIMT = sgr.SGR_PATH_SIMT
TC = sgr.SGR_PATH_W8  # the tensor-core widening kernel


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    torch.cuda.set_device(0)
    sgr.sgr_init(0)
    sgr.sgr_device_error(0, clear=True)
    yield
    assert sgr.sgr_device_error(0) == 0, "a kernel reported a timed-out wait"


def ref(p) -> np.ndarray:
    return oracle.load().gemm_residual_w4(p.A, p.Wq4, p.bs, p.gs, p.R)


def scales_on_device(bs: torch.Tensor) -> torch.Tensor:
    """Block scales on the GPU, each row padded to a multiple of 16 bytes (the
    kernel reads scale rows in 16-byte units)."""
    N, nb = bs.shape
    padded = (nb + 15) // 16 * 16
    buf = torch.full((N, padded), 0x7F, dtype=torch.uint8, device="cuda")  # NaN codes in the padding: never used
    buf[:, :nb].copy_(bs)
    return buf[:, :nb]


def codes_on_device(Wq4: torch.Tensor) -> torch.Tensor:
    """Codes on the GPU, rows padded to a multiple of 16 bytes when K/2 is
    not (the row stride must be, the row length need not)."""
    N, half = Wq4.shape
    if half % 16 == 0:
        return Wq4.cuda()
    buf = torch.zeros((N, (half + 15) // 16 * 16), dtype=torch.uint8, device="cuda")
    buf[:, :half].copy_(Wq4)
    return buf[:, :half]


def run(p, **cfg):
    A, Wq4, bs, R = p.A.cuda(), codes_on_device(p.Wq4), scales_on_device(p.bs), p.R.cuda()
    Y = torch.full_like(R, float("nan"))
    sgr.skinny_gemm_residual_w4(A, Wq4, bs, p.gs, R, Y, config=sgr.make_config(**cfg) if cfg else None)
    torch.cuda.synchronize()
    return bits(Y)


def codes_problem(M, N, K, seed, scale_mask=0x7F):
    """Every code pair, random positive block scales (subnormal to 448), a
    non-power-of-two tensor scale."""
    A = inputs.random_bf16_bits((M, K), seed, lo_exp=-3, hi_exp=2)
    Wq4 = inputs.random_e2m1_bytes((N, K // 2), seed + 1)
    bs = inputs.random_e4m3_codes((N, (K + 15) // 16), seed + 2) & scale_mask
    bs = torch.where(bs == 0x7F, bs - 1, bs)
    gs = float(inputs.random_scales(1, seed + 3, lo_exp=-8, hi_exp=-4)[0])
    R = inputs.random_bf16_bits((M, N), seed + 4, lo_exp=-3, hi_exp=3)
    return inputs.ProblemW4(A, Wq4, bs, gs, R, seed)


@pytest.mark.parametrize("M,N,K", [(1, 8, 32), (1, 520, 1056), (2, 304, 64), (3, 1000, 3584), (4, 2056, 992),
                                   (5, 776, 512), (8, 8, 7168), (9, 264, 1024), (16, 1032, 2048)])
def test_w4_small_shapes(M, N, K):
    """Ragged in every dimension: M across the 4-token pass, N not a multiple
    of the rows per CTA, K with a partial last scale row (66 blocks at K =
    1056, read as 80 bytes) and the largest K (7168)."""
    p = inputs.make_problem_w4(M, N, K, seed=M * 13 + N + K)
    compare(run(p), ref(p), f"w4 {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(1, 512, 256), (4, 1024, 3584), (7, 264, 640)])
def test_w4_every_code_and_scale(M, N, K):
    p = codes_problem(M, N, K, seed=M + N + K)
    compare(run(p), ref(p), f"w4 codes {M}x{N}x{K}")


def test_w4_subnormal_block_scales():
    """Only zero and subnormal block scales (exponent field 0): products down
    to 0.5 * 2^-9, where the FP16 product must still be exact."""
    p = codes_problem(3, 512, 1024, seed=41, scale_mask=0x07)
    compare(run(p), ref(p), "w4 subnormal scales")


@pytest.mark.parametrize("seed", [0, 1])
@pytest.mark.parametrize("M", [1, 2, 4, 8, 16])
def test_w4_full_size_m_sweep(M, seed):
    """The decode sweep at the latent-MoE shape, every element."""
    p = inputs.make_problem_w4(M, N_FULL, K_FULL, seed=seed * 100 + M)
    m = compare(run(p), ref(p), f"w4 M={M} seed={seed}")
    assert m["cosine"] > 0.999


def test_w4_down_projection():
    p = inputs.make_problem_w4(4, 3584, 7168, seed=5)
    compare(run(p), ref(p), "w4 down-projection")


W4_CONFIGS = [
    dict(path=SIMT, ctas_per_sm=1, rows_per_stage=1, stages=2),
    dict(path=SIMT, ctas_per_sm=2, rows_per_stage=4, stages=3),
    dict(path=SIMT, ctas_per_sm=1, rows_per_stage=8, stages=6),
    dict(path=SIMT, ctas_per_sm=3, rows_per_stage=2, stages=8),
]


@pytest.mark.parametrize("cfg", W4_CONFIGS, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items() if k != "path"))
@pytest.mark.parametrize("M", [1, 3, 6])
def test_w4_configs(cfg, M):
    p = inputs.make_problem_w4(M, 2056, 1024, seed=31 + M)
    compare(run(p, **cfg), ref(p), f"w4 M={M} {cfg}")


@pytest.mark.parametrize("M", [1, 2, 3, 4, 8, 16])
def test_w4_both_kernels_full_size(M):
    """The CUDA-core and tensor-core kernels, forced, at the latent-MoE
    shape: every element of each against the oracle."""
    p = inputs.make_problem_w4(M, N_FULL, K_FULL, seed=200 + M)
    want = ref(p)
    compare(run(p, path=SIMT), want, f"w4 simt M={M}")
    compare(run(p, path=TC), want, f"w4 tensor core M={M}")


@pytest.mark.parametrize("M,N,K", [(1, 8, 8), (3, 520, 1000), (5, 776, 72), (17, 1024, 2056), (40, 2056, 3584),
                                   (64, 1024, 1024), (100, 264, 3600), (256, 1032, 512)])
def test_w4_tensor_core_ragged_and_wide(M, N, K):
    """The tensor-core kernel on shapes the CUDA-core kernel cannot take (K
    not a multiple of 32, padded code rows) and at 17-256 tokens in one
    launch (token tiles of 32-256)."""
    p = inputs.make_problem_w4(M, N, K, seed=M * 3 + N + K)
    compare(run(p, path=TC), ref(p), f"w4 tc {M}x{N}x{K}")


TC_CONFIGS = [
    dict(path=TC, k_blocks_per_stage=4, stages=2),
    dict(path=TC, k_blocks_per_stage=4, stages=6, prefetch_stages=4),
    dict(path=TC, k_blocks_per_stage=8, stages=2),
    dict(path=TC, k_blocks_per_stage=8, stages=3, prefetch_stages=3),
    dict(path=TC, k_blocks_per_stage=8, stages=2, rows_per_stage=32),
    dict(path=TC, k_blocks_per_stage=4, stages=4, token_tile=32),
]


@pytest.mark.parametrize("cfg", TC_CONFIGS, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items() if k != "path"))
@pytest.mark.parametrize("M", [1, 7, 16])
def test_w4_tensor_core_configs(cfg, M):
    p = inputs.make_problem_w4(M, 2056, 1032, seed=41 + M)
    compare(run(p, **cfg), ref(p), f"w4 tc M={M} {cfg}")


def test_w4_tensor_core_every_code_and_subnormal_scales():
    p = codes_problem(6, 512, 1024, seed=43)
    compare(run(p, path=TC), ref(p), "w4 tc codes")
    q = codes_problem(3, 512, 1024, seed=44, scale_mask=0x07)
    compare(run(q, path=TC), ref(q), "w4 tc subnormal scales")


def test_w4_integer_inputs_exact():
    """Integer activations and residuals, codes of integer value (0, 1, 2, 3,
    4, 6 and their negatives), block scales 1 or 2, gs = 1: every partial sum is an
    exact integer, so the result must equal the integer sum rounded once."""
    M, N, K = 4, 1024, 1024
    A = inputs.integer_bf16((M, K), -3, 3, 51)
    R = inputs.integer_bf16((M, N), -16, 16, 52)
    g = torch.Generator().manual_seed(53)
    nib = torch.tensor([0, 2, 4, 5, 6, 7, 10, 12, 13, 14, 15], dtype=torch.int64)  # integer-valued codes
    codes = nib[torch.randint(0, len(nib), (N, K), generator=g)]
    Wq4 = (codes[:, 0::2] | (codes[:, 1::2] << 4)).to(torch.uint8)
    bs = torch.where(torch.rand((N, K // 16), generator=g) < 0.5, 0x38, 0x40).to(torch.uint8)  # 1.0 or 2.0
    table = torch.tensor([0, 0.5, 1, 1.5, 2, 3, 4, 6, 0, -0.5, -1, -1.5, -2, -3, -4, -6], dtype=torch.float64)
    Wv = table[codes] * torch.where(bs == 0x38, 1.0, 2.0).to(torch.float64).repeat_interleave(16, dim=1)
    want = A.to(torch.float64) @ Wv.T + R.to(torch.float64)
    assert want.abs().max() < 2 ** 24 and torch.equal(Wv, Wv.round())
    Y = sgr.skinny_gemm_residual_w4(A.cuda(), Wq4.cuda(), scales_on_device(bs), 1.0, R.cuda())
    torch.cuda.synchronize()
    assert torch.equal(Y.cpu(), want.to(torch.float32).to(torch.bfloat16))


def test_w4_float8_scale_dtype_and_deterministic():
    p = inputs.make_problem_w4(3, 1024, 2048, seed=61)
    y1 = run(p)
    A, Wq4, R = p.A.cuda(), p.Wq4.cuda(), p.R.cuda()
    bs = scales_on_device(p.bs).view(torch.float8_e4m3fn)
    Y = sgr.skinny_gemm_residual_w4(A, Wq4, bs, p.gs, R)
    torch.cuda.synchronize()
    assert np.array_equal(y1, bits(Y)) and np.array_equal(y1, run(p))


def test_w4_strided_padded_and_in_place():
    """A a column slice of a wider buffer, code rows padded (row stride above
    K/2), scale rows padded beyond 16 bytes, R and Y the same column slice of
    a wider buffer (in-place update); the rest of the buffers untouched."""
    M, N, K = 5, 1024, 1024
    p = inputs.make_problem_w4(M, N, K, seed=71)
    Abig = torch.zeros((M, K + 64), dtype=torch.bfloat16, device="cuda")
    A = Abig[:, 64:]
    A.copy_(p.A)
    Wbig = torch.zeros((N, K // 2 + 48), dtype=torch.uint8, device="cuda")
    Wq4 = Wbig[:, 16:16 + K // 2]
    Wq4.copy_(p.Wq4)
    Sbig = torch.zeros((N, 128), dtype=torch.uint8, device="cuda")
    bs = Sbig[:, 32:32 + K // 16]
    bs.copy_(p.bs)
    big = torch.full((M, N + 512), 3.0, dtype=torch.bfloat16, device="cuda")
    RY = big[:, 256:256 + N]
    RY.copy_(p.R)
    sgr.skinny_gemm_residual_w4(A, Wq4, bs, p.gs, RY, RY)
    torch.cuda.synchronize()
    compare(bits(RY), ref(p), "w4 strided in-place")
    assert torch.all(big[:, :256] == 3.0) and torch.all(big[:, 256 + N:] == 3.0)


def test_w4_graph_replay_and_pdl_chain():
    """Three dependent NVFP4 layers (A_i = Y_{i-1}[:, :K]) captured in one
    CUDA graph with programmatic dependent launch, against the oracle layer
    by layer on the GPU's own intermediate outputs."""
    M, N, K = 4, 2048, 1024
    probs = [inputs.make_problem_w4(M, N, K, seed=80 + i) for i in range(3)]
    dW = [q.Wq4.cuda() for q in probs]
    dS = [scales_on_device(q.bs) for q in probs]
    dR = [q.R.cuda() for q in probs]
    A0 = probs[0].A.cuda()
    Ys = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    stream = torch.cuda.Stream()

    def chain():
        for i in range(3):
            A = A0 if i == 0 else Ys[i - 1][:, :K]
            sgr.skinny_gemm_residual_w4(A, dW[i], dS[i], probs[i].gs, dR[i], Ys[i], stream=stream)

    with torch.cuda.stream(stream):
        chain()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        chain()
    for Y in Ys:
        Y.fill_(float("nan"))
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    A = probs[0].A
    for i in range(3):
        q = probs[i]
        want = oracle.load().gemm_residual_w4(A, q.Wq4, q.bs, q.gs, q.R)
        compare(bits(Ys[i]), want, f"w4 chain layer {i}")
        A = Ys[i].cpu()[:, :K]


def test_w4_empty_and_k0():
    R = inputs.make_rows(3, 64, seed=1).cuda()
    Y = sgr.skinny_gemm_residual_w4(torch.empty((3, 0), dtype=torch.bfloat16, device="cuda"),
                                    torch.empty((64, 0), dtype=torch.uint8, device="cuda"),
                                    torch.empty((64, 0), dtype=torch.uint8, device="cuda"), 1.0, R)
    torch.cuda.synchronize()
    assert torch.equal(Y, R)


def test_w4_rejects():
    p = inputs.make_problem_w4(2, 256, 1024, seed=2)
    A, Wq4, bs, R = p.A.cuda(), p.Wq4.cuda(), scales_on_device(p.bs), p.R.cuda()
    for cfg in (dict(path=sgr.SGR_PATH_TILE), dict(path=sgr.SGR_PATH_W8S), dict(path=SIMT, stages=1),
                dict(path=SIMT, rows_per_stage=65), dict(path=SIMT, ctas_per_sm=9), dict(k_split=2),
                dict(path=TC, k_blocks_per_stage=2), dict(path=TC, k_blocks_per_stage=6), dict(path=TC, stages=17),
                dict(path=TC, ctas_per_sm=2), dict(path=TC, token_tile=8)):
        with pytest.raises(sgr.SgrError) as e:
            sgr.skinny_gemm_residual_w4(A, Wq4, bs, p.gs, R, config=sgr.make_config(**cfg))
        assert e.value.status == sgr.SGR_ERR_UNSUPPORTED, cfg
    q = inputs.make_problem_w4(1, 64, 48, seed=3)  # K = 48: not whole 32-code vectors
    with pytest.raises(sgr.SgrError) as e:
        sgr.skinny_gemm_residual_w4(q.A.cuda(), codes_on_device(q.Wq4), scales_on_device(q.bs), q.gs, q.R.cuda(),
                                    config=sgr.make_config(path=SIMT))
    assert e.value.status == sgr.SGR_ERR_UNSUPPORTED
    y = sgr.skinny_gemm_residual_w4(q.A.cuda(), codes_on_device(q.Wq4), scales_on_device(q.bs), q.gs, q.R.cuda())
    torch.cuda.synchronize()  # the library's choice takes the tensor-core kernel there
    compare(bits(y), ref(q), "w4 K = 48 (automatic path)")
