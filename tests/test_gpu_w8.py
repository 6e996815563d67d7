"""GPU parity of the FP8-weight kernel (skinny_gemm_residual_w8) against the
CPU oracle's low-bit variant, element by element on the same seeded inputs."""
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
    """Codes on the GPU; rows padded to a multiple of 16 bytes when K is not
    (the row stride of the code matrix must be, the row length need not)."""
    N, K = Wq.shape
    if K % 16 == 0:
        return Wq.cuda()
    buf = torch.zeros((N, (K + 15) // 16 * 16), dtype=torch.uint8, device="cuda")
    buf[:, :K].copy_(Wq)
    return buf[:, :K]


def run(p, **cfg):
    A, Wq, sc, R = p.A.cuda(), codes_on_device(p.Wq), p.scale.cuda(), p.R.cuda()
    Y = torch.full_like(R, float("nan"))
    sgr.skinny_gemm_residual_w8(A, Wq, sc, R, Y, config=sgr.make_config(**cfg) if cfg else None)
    torch.cuda.synchronize()
    return bits(Y)


def codes_problem(M, N, K, seed, mask=0xFF):
    """Every kind of code (zero, subnormal, normal, both signs), random scales."""
    A = inputs.random_bf16_bits((M, K), seed, lo_exp=-3, hi_exp=2)
    Wq = inputs.random_e4m3_codes((N, K), seed + 1) & mask
    sc = inputs.random_scales(N, seed + 2, lo_exp=-14, hi_exp=-8)
    R = inputs.random_bf16_bits((M, N), seed + 3, lo_exp=-3, hi_exp=3)
    return inputs.ProblemW8(A, Wq, sc, R, seed)


SMALL = [(1, 520, 264), (3, 7168, 64), (4, 2056, 3584), (5, 304, 8), (7, 1512, 1800), (16, 2056, 3584),
         (16, 8, 3584), (1, 8, 8), (13, 152, 1792), (17, 200, 136), (40, 1000, 1032), (100, 1024, 520),
         (250, 264, 1000), (256, 392, 264)]


@pytest.mark.parametrize("M,N,K", SMALL)
def test_w8_small_shapes(M, N, K):
    p = inputs.make_problem_w8(M, N, K, seed=M * 7 + N + K)
    compare(run(p), ref(p), f"w8 {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(1, 264, 200), (4, 1024, 520), (16, 152, 1032), (33, 304, 264)])
def test_w8_every_kind_of_code(M, N, K):
    """Uniformly random codes: one in 16 has a zero exponent field, so most
    32-code groups take the exact slow widening path."""
    p = codes_problem(M, N, K, seed=M + N + K)
    compare(run(p), ref(p), f"w8 random codes {M}x{N}x{K}")


def test_w8_subnormal_and_zero_codes():
    """Only exponent fields 0 and 1 (zero, subnormals, the smallest binade)."""
    p = codes_problem(8, 1024, 1024, seed=5, mask=0x8F)
    p.scale.mul_(2.0 ** 12)
    compare(run(p), ref(p), "w8 subnormal codes")


@pytest.mark.parametrize("M", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("seed", [0, 1])
def test_w8_full_size_m_sweep(M, seed):
    p = inputs.make_problem_w8(M, N_FULL, K_FULL, seed=seed)
    compare(run(p), ref(p), f"w8 M={M} seed={seed}")


@pytest.mark.parametrize("M", [32, 64, 128])
def test_w8_full_size_transition(M):
    p = inputs.make_problem_w8(M, N_FULL, K_FULL, seed=M)
    compare(run(p), ref(p), f"w8 M={M}")


def test_w8_full_size_m256_sampled():
    M = 256
    p = inputs.make_problem_w8(M, N_FULL, K_FULL, seed=9)
    got = run(p)
    rng = np.random.default_rng(M)
    ms = np.concatenate([rng.integers(0, M, 4000), np.zeros(N_FULL, int), np.full(N_FULL, M - 1)])
    ns = np.concatenate([rng.integers(0, N_FULL, 4000), np.arange(N_FULL), np.arange(N_FULL)])
    want = oracle.load().sample_w8(p.A, p.Wq, p.scale, p.R, ms, ns)
    compare(got[ms, ns], want, "w8 M=256 sampled")


def test_w8_down_projection():
    p = inputs.make_problem_w8(8, K_FULL, N_FULL, seed=3)
    compare(run(p), ref(p), "w8 down-projection N=3584 K=7168")


CONFIGS = [
    dict(k_blocks_per_stage=2, stages=2),
    dict(k_blocks_per_stage=2, stages=8),
    dict(k_blocks_per_stage=4, stages=3),
    dict(k_blocks_per_stage=4, stages=6, prefetch_stages=2),
    dict(k_blocks_per_stage=4, stages=12, prefetch_stages=8),
    dict(k_blocks_per_stage=8, stages=2),
    dict(k_blocks_per_stage=8, stages=4, prefetch_stages=4),
    dict(k_blocks_per_stage=6, stages=3),
    dict(k_blocks_per_stage=4, stages=4, token_tile=32),
    dict(rows_per_stage=32, k_blocks_per_stage=4, stages=4),
    dict(rows_per_stage=64, k_blocks_per_stage=4, stages=3),
    dict(rows_per_stage=24, k_blocks_per_stage=4, stages=3),
    dict(rows_per_stage=8, k_blocks_per_stage=8, stages=3),
    dict(rows_per_stage=128, k_blocks_per_stage=2, stages=4),
]


@pytest.mark.parametrize("cfg", CONFIGS, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
@pytest.mark.parametrize("M", [1, 9, 16])
def test_w8_configs(cfg, M):
    p = inputs.make_problem_w8(M, N_FULL, K_FULL, seed=71 + M)
    compare(run(p, path=sgr.SGR_PATH_W8, **cfg), ref(p), f"w8 M={M} {cfg}")


def test_w8_integer_inputs_exact():
    """Small-integer codes, scale 1, integer A and R: every partial sum is an
    exact integer in FP32, so the result equals the int64 product exactly."""
    M, N, K = 16, 2048, 1024
    A = inputs.integer_bf16((M, K), -2, 2, 4)
    vals = inputs.integer_bf16((N, K), -8, 8, 5).to(torch.float32)
    Wq = vals.to(torch.float8_e4m3fn).view(torch.uint8)
    assert torch.equal(Wq.view(torch.float8_e4m3fn).to(torch.float32), vals)
    R = inputs.integer_bf16((M, N), -8, 8, 6)
    want = A.to(torch.int64) @ vals.to(torch.int64).T + R.to(torch.int64)
    assert want.abs().max() < 2 ** 24
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    sgr.skinny_gemm_residual_w8(A.cuda(), Wq.cuda(), torch.ones(N, device="cuda"), R.cuda(), Y)
    torch.cuda.synchronize()
    assert np.array_equal(bits(Y), bits(want.to(torch.bfloat16)))


def test_w8_float8_dtype_and_deterministic():
    p = inputs.make_problem_w8(6, N_FULL, K_FULL, seed=44)
    y1 = run(p)
    A, R = p.A.cuda(), p.R.cuda()
    Y2 = torch.empty_like(R)
    sgr.skinny_gemm_residual_w8(A, p.Wq.cuda().view(torch.float8_e4m3fn), p.scale.cuda(), R, Y2,
                                flags=sgr.SGR_FLAG_NO_PDL)
    torch.cuda.synchronize()
    assert np.array_equal(y1, bits(Y2))


def test_w8_strided_padded_and_in_place():
    M, N, K = 6, 2048, 1024
    p = inputs.make_problem_w8(M, N, K, seed=55)
    Abig = torch.zeros((M, K + 128), dtype=torch.bfloat16, device="cuda")
    A = Abig[:, 64:64 + K]
    A.copy_(p.A)
    Wbig = torch.zeros((N, K + 48), dtype=torch.uint8, device="cuda")  # code rows padded to K + 48 bytes
    Wq = Wbig[:, 16:16 + K]
    Wq.copy_(p.Wq)
    RY = torch.zeros((M, N + 64), dtype=torch.bfloat16, device="cuda")
    RY[:, 8:8 + N].copy_(p.R)
    view = RY[:, 8:8 + N]
    sgr.skinny_gemm_residual_w8(A, Wq, p.scale.cuda(), view, view)
    torch.cuda.synchronize()
    compare(bits(view), ref(p), "w8 strided, padded codes, in place")
    assert torch.all(RY[:, :8] == 0) and torch.all(RY[:, 8 + N:] == 0)


def test_w8_graph_replays():
    probs = [inputs.make_problem_w8(4, N_FULL, K_FULL, seed=60 + s) for s in range(3)]
    dev = [[t.cuda() for t in (q.A, q.Wq, q.scale, q.R)] for q in probs]
    outs = [torch.empty_like(d[3]) for d in dev]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for (A, Wq, sc, R), Y in zip(dev, outs):
            sgr.skinny_gemm_residual_w8(A, Wq, sc, R, Y)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = [bits(Y) for Y in outs]
    for Y in outs:
        Y.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for (A, Wq, sc, R), Y in zip(dev, outs):
            sgr.skinny_gemm_residual_w8(A, Wq, sc, R, Y)
    for _ in range(10):
        g.replay()
    torch.cuda.synchronize()
    for e, Y in zip(eager, outs):
        assert np.array_equal(e, bits(Y))
    compare(eager[2], ref(probs[2]), "w8 graph")


def test_w8_chained_layers_with_pdl():
    """Each call's A is the previous call's Y (N = K): launched back to back
    with programmatic dependent launch, every layer must see the finished
    output of the one before."""
    D, M, L = 1024, 4, 6
    ps = [inputs.make_problem_w8(M, D, D, seed=80 + i) for i in range(L)]
    x = ps[0].A.cuda()
    R = [q.R.cuda() for q in ps]
    Wq = [q.Wq.cuda() for q in ps]
    sc = [q.scale.cuda() for q in ps]
    ys = [torch.empty((M, D), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    inp = x
    for i in range(L):
        sgr.skinny_gemm_residual_w8(inp, Wq[i], sc[i], R[i], ys[i])
        inp = ys[i]
    torch.cuda.synchronize()
    a = ps[0].A
    for i in range(L):
        want = oracle.load().gemm_residual_w8(a, ps[i].Wq, ps[i].scale, ps[i].R)
        got = bits(ys[i])
        compare(got, want, f"w8 chain layer {i}")
        a = oracle.from_bits(got)  # the next layer consumes the GPU's own rounded output


def test_w8_empty_and_k0():
    R = torch.randn((3, 64), device="cuda").to(torch.bfloat16)
    Y = torch.zeros_like(R)
    A = torch.empty((3, 0), dtype=torch.bfloat16, device="cuda")
    Wq = torch.empty((64, 0), dtype=torch.uint8, device="cuda")
    sgr.skinny_gemm_residual_w8(A, Wq, torch.ones(64, device="cuda"), R, Y)
    torch.cuda.synchronize()
    assert torch.equal(Y, R)
    A0 = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    W0 = torch.zeros((64, 64), dtype=torch.uint8, device="cuda")
    R0 = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    sgr.skinny_gemm_residual_w8(A0, W0, torch.ones(64, device="cuda"), R0)


def test_w8_rejects_bad_config():
    p = inputs.make_problem_w8(20, 256, 256, seed=1)
    A, Wq, sc, R = p.A.cuda(), p.Wq.cuda(), p.scale.cuda(), p.R.cuda()
    for cfg in (dict(path=sgr.SGR_PATH_TC_ROWS), dict(path=sgr.SGR_PATH_TILE), dict(path=sgr.SGR_PATH_W8, token_tile=16),
                dict(path=sgr.SGR_PATH_W8, k_blocks_per_stage=3), dict(path=sgr.SGR_PATH_W8, stages=17),
                dict(path=sgr.SGR_PATH_W8, rows_per_stage=20), dict(path=sgr.SGR_PATH_W8, tile_n=128),
                dict(path=sgr.SGR_PATH_W8, prefetch_stages=9), dict(path=sgr.SGR_PATH_W8, stages=8, prefetch_stages=1)):
        with pytest.raises(sgr.SgrError) as e:
            sgr.skinny_gemm_residual_w8(A, Wq, sc, R, config=sgr.make_config(**cfg))
        assert e.value.status == sgr.SGR_ERR_UNSUPPORTED
    with pytest.raises(sgr.SgrError) as e:  # more than 256 tokens
        q = inputs.make_problem_w8(257, 256, 256, seed=2)
        sgr.skinny_gemm_residual_w8(q.A.cuda(), q.Wq.cuda(), q.scale.cuda(), q.R.cuda())
    assert e.value.status == sgr.SGR_ERR_UNSUPPORTED


# ------------------------------------------------------------------ CUDA-core FP8 kernel (M <= 8)
SIMT = sgr.SGR_PATH_SIMT


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8])
def test_w8_simt_full_size(M):
    p = inputs.make_problem_w8(M, N_FULL, K_FULL, seed=300 + M)
    compare(run(p, path=SIMT), ref(p), f"w8 simt M={M}")


@pytest.mark.parametrize("M,N,K", [(1, 520, 272), (3, 304, 16), (4, 2056, 3584), (8, 152, 1792), (2, 8, 7168),
                                   (1, 1000, 14336), (7, 1512, 1808)])
def test_w8_simt_small_shapes(M, N, K):
    p = codes_problem(M, N, K, seed=M + N + K + 1)
    compare(run(p, path=SIMT), ref(p), f"w8 simt random codes {M}x{N}x{K}")


def test_w8_simt_subnormal_codes():
    p = codes_problem(4, 1024, 1024, seed=6, mask=0x8F)
    p.scale.mul_(2.0 ** 12)
    compare(run(p, path=SIMT), ref(p), "w8 simt subnormal codes")


SIMT_CONFIGS = [dict(ctas_per_sm=1, rows_per_stage=4, stages=4), dict(ctas_per_sm=2, rows_per_stage=1, stages=8),
                dict(ctas_per_sm=3, rows_per_stage=2, stages=2), dict(ctas_per_sm=1, rows_per_stage=16, stages=3)]


@pytest.mark.parametrize("cfg", SIMT_CONFIGS, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
@pytest.mark.parametrize("M", [1, 4])
def test_w8_simt_configs(cfg, M):
    p = inputs.make_problem_w8(M, N_FULL, K_FULL, seed=400 + M)
    compare(run(p, path=SIMT, **cfg), ref(p), f"w8 simt M={M} {cfg}")


def test_w8_simt_strided_in_place():
    M, N, K = 3, 2048, 1024
    p = inputs.make_problem_w8(M, N, K, seed=57)
    Abig = torch.zeros((M, K + 64), dtype=torch.bfloat16, device="cuda")
    A = Abig[:, 32:32 + K]
    A.copy_(p.A)
    RY = torch.zeros((M, N + 16), dtype=torch.bfloat16, device="cuda")
    view = RY[:, 8:8 + N]
    view.copy_(p.R)
    sgr.skinny_gemm_residual_w8(A, p.Wq.cuda(), p.scale.cuda(), view, view,
                                config=sgr.make_config(path=SIMT))
    torch.cuda.synchronize()
    compare(bits(view), ref(p), "w8 simt strided in place")


def test_w8_auto_small_m_matches_tensor_core_path():
    """AUTO picks the FP8 tensor-core kernel with split activations for M = 1;
    it, the widening tensor-core kernel and the CUDA-core kernel all agree
    with the oracle."""
    p = inputs.make_problem_w8(1, N_FULL, K_FULL, seed=58)
    want = ref(p)
    compare(run(p), want, "w8 auto M=1")
    compare(run(p, path=sgr.SGR_PATH_W8S), want, "w8 split FP8 M=1")
    compare(run(p, path=sgr.SGR_PATH_W8), want, "w8 tensor-core M=1")
    compare(run(p, path=sgr.SGR_PATH_SIMT), want, "w8 CUDA-core M=1")


@pytest.mark.parametrize("M", [3, 6, 12])
def test_w8_auto_matches_oracle(M):
    """AUTO at token counts served by the split-activation kernel's two
    instances (3: A in registers; 6: A read per stage) and by the widening
    kernel (12)."""
    p = inputs.make_problem_w8(M, N_FULL, K_FULL, seed=60 + M)
    compare(run(p), ref(p), f"w8 auto M={M}")


def test_w8_simt_rejects():
    p = inputs.make_problem_w8(9, 256, 256, seed=3)
    with pytest.raises(sgr.SgrError) as e:  # more than 8 tokens
        sgr.skinny_gemm_residual_w8(p.A.cuda(), p.Wq.cuda(), p.scale.cuda(), p.R.cuda(),
                                    config=sgr.make_config(path=SIMT))
    assert e.value.status == sgr.SGR_ERR_UNSUPPORTED
    q = inputs.make_problem_w8(2, 256, 264, seed=4)  # K not a multiple of 16 (padded code rows)
    with pytest.raises(sgr.SgrError) as e:
        sgr.skinny_gemm_residual_w8(q.A.cuda(), codes_on_device(q.Wq), q.scale.cuda(), q.R.cuda(),
                                    config=sgr.make_config(path=SIMT))
    assert e.value.status == sgr.SGR_ERR_UNSUPPORTED
    r = inputs.make_problem_w8(2, 256, 256, seed=5)
    with pytest.raises(sgr.SgrError) as e:  # a tile-only field
        sgr.skinny_gemm_residual_w8(r.A.cuda(), r.Wq.cuda(), r.scale.cuda(), r.R.cuda(),
                                    config=sgr.make_config(path=SIMT, token_tile=16))
    assert e.value.status == sgr.SGR_ERR_UNSUPPORTED
