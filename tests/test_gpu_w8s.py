"""GPU parity of the FP8-weight kernel on the FP8 tensor-core path
(skinny_gemm_residual_w8 with SGR_PATH_W8S: codes straight into kind::f8f6f4
MMAs, activations split into two E4M3 parts under a per-token power-of-two
scale) against the CPU oracle's low-bit variant."""
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
W8S = sgr.SGR_PATH_W8S


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
    return oracle.load().gemm_residual_w8(p.A, p.Wq, p.scale, p.R)


def codes_on_device(Wq: torch.Tensor) -> torch.Tensor:
    """Codes on the GPU, rows padded to a multiple of 16 bytes when K is not."""
    N, K = Wq.shape
    if K % 16 == 0:
        return Wq.cuda()
    buf = torch.zeros((N, (K + 15) // 16 * 16), dtype=torch.uint8, device="cuda")
    buf[:, :K].copy_(Wq)
    return buf[:, :K]


def run(p, **cfg):
    A, Wq, sc, R = p.A.cuda(), codes_on_device(p.Wq), p.scale.cuda(), p.R.cuda()
    Y = torch.full_like(R, float("nan"))
    sgr.skinny_gemm_residual_w8(A, Wq, sc, R, Y, config=sgr.make_config(path=W8S, **cfg))
    torch.cuda.synchronize()
    return bits(Y)


def codes_problem(M, N, K, seed, a_lo=-3, a_hi=2):
    """Every kind of code (zero, subnormal, normal, both signs), random scales."""
    A = inputs.random_bf16_bits((M, K), seed, lo_exp=a_lo, hi_exp=a_hi)
    Wq = inputs.random_e4m3_codes((N, K), seed + 1)
    sc = inputs.random_scales(N, seed + 2, lo_exp=-14, hi_exp=-8)
    R = inputs.random_bf16_bits((M, N), seed + 3, lo_exp=-3, hi_exp=3)
    return inputs.ProblemW8(A, Wq, sc, R, seed)


# Ragged: K not a multiple of the 128-code block (partial last block, odd
# block counts that leave a padding block in the last MMA window), N not a
# multiple of the slab, M = 1 .. 16 on both token widths (8 and 16).
SMALL = [(1, 520, 264), (3, 7168, 64), (4, 2056, 3584), (5, 304, 8), (7, 1512, 1800), (8, 1000, 136),
         (9, 2056, 3584), (16, 8, 3584), (1, 8, 8), (13, 152, 1792), (16, 1000, 1032), (12, 392, 392)]


@pytest.mark.parametrize("M,N,K", SMALL)
def test_w8s_small_shapes(M, N, K):
    p = inputs.make_problem_w8(M, N, K, seed=M * 11 + N + K)
    compare(run(p), ref(p), f"w8s {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(4, 2056, 1032), (16, 1000, 3584), (1, 264, 264)])
def test_w8s_every_kind_of_code(M, N, K):
    p = codes_problem(M, N, K, seed=5 * M + K)
    compare(run(p), ref(p), f"w8s codes {M}x{N}x{K}")


@pytest.mark.parametrize("M", [1, 2, 3, 4, 6, 8, 16])
@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_w8s_full_size_m_sweep(M, seed):
    p = inputs.make_problem_w8(M, N_FULL, K_FULL, seed=seed)
    m = compare(run(p), ref(p), f"w8s M={M} seed={seed}")
    assert m["cosine"] > 0.999


@pytest.mark.parametrize("M", [1, 4, 8])
def test_w8s_down_projection(M):
    """K = 7168 (the down-projection) with up to 8 tokens."""
    p = inputs.make_problem_w8(M, K_FULL, N_FULL, seed=30 + M)
    compare(run(p), ref(p), f"w8s down M={M}")


def test_w8s_activation_outliers_within_tolerance():
    """Rows whose largest activations are up to 2^12 times the typical one
    (massive activation outliers in a few channels): every value is within
    2^13 of its row's maximum, so the split is exact and the result is within
    the parity gate."""
    M, N, K = 16, 2048, 3584
    p = inputs.make_problem_w8(M, N, K, seed=71)
    A = p.A.to(torch.float32)
    A[:, 17] *= 4096.0
    A[:, 1000] *= -2048.0
    A[3, 5] = 1024.0
    p = inputs.ProblemW8(A.to(torch.bfloat16), p.Wq, p.scale, p.R, 71)
    compare(run(p), ref(p), "w8s outliers")


def test_w8s_beyond_exact_range_error_bound():
    """A row whose maximum is 2^20 times its typical value: the values more
    than 2^13 below the maximum are rounded, each by less than 2^-21 of the
    row's maximum, and the result obeys that bound (summed over k with the
    weights' magnitudes) on top of the parity gate."""
    M, N, K = 4, 1024, 2048
    p = inputs.make_problem_w8(M, N, K, seed=77)
    A = p.A.to(torch.float32)
    A[2, 5] = 2.0 ** 20
    p = inputs.ProblemW8(A.to(torch.bfloat16), p.Wq, p.scale, p.R, 77)
    got = run(p)
    want = ref(p)
    from parity import f64
    g, r = f64(got), f64(want)
    wv = p.Wq.view(torch.float8_e4m3fn).to(torch.float64).numpy() * p.scale.to(torch.float64).numpy()[:, None]
    amax = np.abs(A.to(torch.bfloat16).to(torch.float64).numpy()).max(axis=1)
    bound = (np.abs(wv).sum(axis=1)[None, :] * amax[:, None]) * 2.0 ** -21
    assert np.all(np.abs(g - r) <= 1e-2 * np.abs(r) + 2e-2 + bound), "error beyond the stated bound"
    other = [0, 1, 3]  # rows within the exact range pass the plain gate
    compare(got[other], want[other], "w8s rows within range")


def test_w8s_wide_exponent_spread():
    """Activations spread over 16 binades in every row."""
    p = codes_problem(8, 1024, 2048, seed=72, a_lo=-10, a_hi=5)
    compare(run(p), ref(p), "w8s wide spread")


def test_w8s_zero_and_subnormal_activation_rows():
    M, N, K = 6, 512, 512
    p = inputs.make_problem_w8(M, N, K, seed=73)
    A = p.A.clone()
    A[1] = 0.0
    A[2] = torch.tensor(2.0 ** -130, dtype=torch.float32).to(torch.bfloat16)  # BF16 subnormals
    A[4, ::3] = 0.0
    p = inputs.ProblemW8(A, p.Wq, p.scale, p.R, 73)
    compare(run(p), ref(p), "w8s zero / subnormal rows")


def test_w8s_integer_inputs_exact():
    """Small-integer codes, scale 1, integer A and R: every product and partial
    sum is an exact integer, so the result equals the int64 product exactly."""
    M, N, K = 16, 2048, 1024
    A = inputs.integer_bf16((M, K), -2, 2, 74)
    vals = inputs.integer_bf16((N, K), -8, 8, 75).to(torch.float32)
    Wq = vals.to(torch.float8_e4m3fn).view(torch.uint8)
    R = inputs.integer_bf16((M, N), -8, 8, 76)
    want = A.to(torch.int64) @ vals.to(torch.int64).T + R.to(torch.int64)
    assert want.abs().max() < 2 ** 24
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    sgr.skinny_gemm_residual_w8(A.cuda(), Wq.cuda(), torch.ones(N, device="cuda"), R.cuda(), Y,
                                config=sgr.make_config(path=W8S))
    torch.cuda.synchronize()
    assert np.array_equal(bits(Y), bits(want.to(torch.bfloat16)))


@pytest.mark.parametrize("M,kbps,stages,nt", [(1, 4, 4, 8), (4, 4, 4, 8), (5, 8, 2, 8), (8, 8, 2, 8), (9, 8, 2, 16),
                                               (16, 8, 2, 16)])
def test_w8s_default_configs(M, kbps, stages, nt):
    """The measured defaults at the latent-MoE shape: four stages of four
    128-code blocks while A fits the converters' registers (up to 4 tokens),
    two stages of eight above."""
    c = sgr.sgr_default_config(M, N_FULL, K_FULL, path=W8S)
    assert (c.path, c.k_blocks_per_stage, c.stages, c.token_tile) == (W8S, kbps, stages, nt)


W8S_CONFIGS = [
    dict(k_blocks_per_stage=2, stages=2),
    dict(k_blocks_per_stage=4, stages=3),
    dict(k_blocks_per_stage=8, stages=2),
    dict(k_blocks_per_stage=6, stages=2),
    dict(k_blocks_per_stage=1, stages=8),
    dict(k_blocks_per_stage=4, stages=4, token_tile=16),
]


@pytest.mark.parametrize("cfg", W8S_CONFIGS, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
@pytest.mark.parametrize("M", [1, 9, 16])
def test_w8s_configs(cfg, M):
    p = inputs.make_problem_w8(M, N_FULL, K_FULL, seed=81 + M)
    compare(run(p, **cfg), ref(p), f"w8s M={M} {cfg}")


def test_w8s_strided_padded_and_in_place():
    M, N, K = 6, 2048, 1024
    p = inputs.make_problem_w8(M, N, K, seed=56)
    Abig = torch.zeros((M, K + 128), dtype=torch.bfloat16, device="cuda")
    A = Abig[:, 64:64 + K]
    A.copy_(p.A)
    Wbig = torch.zeros((N, K + 48), dtype=torch.uint8, device="cuda")  # code rows padded to K + 48 bytes
    Wq = Wbig[:, 16:16 + K]
    Wq.copy_(p.Wq)
    RY = torch.zeros((M, N + 64), dtype=torch.bfloat16, device="cuda")
    RY[:, 8:8 + N].copy_(p.R)
    view = RY[:, 8:8 + N]
    sgr.skinny_gemm_residual_w8(A, Wq, p.scale.cuda(), view, view, config=sgr.make_config(path=W8S))
    torch.cuda.synchronize()
    compare(bits(view), ref(p), "w8s strided, padded codes, in place")
    assert torch.all(RY[:, :8] == 0) and torch.all(RY[:, 8 + N:] == 0)


def test_w8s_chained_layers_with_pdl_graph():
    """Layer i reads layer i-1's output as its activations, four layers in one
    CUDA graph with programmatic dependent launch."""
    M, D, L = 4, 2048, 4
    ps = [inputs.make_problem_w8(M, D, D, seed=90 + i) for i in range(L)]
    dev = [(q.Wq.cuda(), q.scale.cuda(), q.R.cuda()) for q in ps]
    A0 = ps[0].A.cuda()
    Ys = [torch.empty((M, D), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    cfg = sgr.make_config(path=W8S)
    s = torch.cuda.Stream()

    def layers():
        for i in range(L):
            Wq, sc, R = dev[i]
            sgr.skinny_gemm_residual_w8(A0 if i == 0 else Ys[i - 1], Wq, sc, R, Ys[i], config=cfg, stream=s)

    with torch.cuda.stream(s):
        layers()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        layers()
    for Y in Ys:
        Y.fill_(float("nan"))
    with torch.cuda.stream(s):
        g.replay()
    s.synchronize()
    A = ps[0].A
    for i in range(L):
        q = ps[i]
        want = oracle.load().gemm_residual_w8(A, q.Wq, q.scale, q.R)
        compare(bits(Ys[i]), want, f"w8s chain layer {i}")
        A = Ys[i].cpu()


def test_w8s_rejects():
    p = inputs.make_problem_w8(17, 256, 256, seed=3)  # more than 16 tokens
    with pytest.raises(sgr.SgrError) as e:
        run(p)
    assert e.value.status == sgr.SGR_ERR_UNSUPPORTED
    q = inputs.make_problem_w8(12, 256, 7168, seed=4)  # 16-token width: K beyond what the converters hold
    with pytest.raises(sgr.SgrError) as e:
        run(q)
    assert e.value.status == sgr.SGR_ERR_UNSUPPORTED
    r = inputs.make_problem_w8(4, 256, 256, seed=5)
    for cfg in (dict(tile_n=128), dict(token_tile=32), dict(stages=9), dict(k_blocks_per_stage=9),
                dict(prefetch_stages=2), dict(token_tile=8, k_blocks_per_stage=4, stages=1)):
        with pytest.raises(sgr.SgrError) as e:
            run(r, **cfg)
        assert e.value.status == sgr.SGR_ERR_UNSUPPORTED, cfg
