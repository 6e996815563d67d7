"""GPU parity: the CUDA path through the C ABI against the CPU oracle,
element by element, on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import skinny_bf16_gemm_residual_gb300 as sgr
from skinny_bf16_gemm_residual_gb300 import inputs
from parity import bits, compare, oracle_full, oracle_problem

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


def run_gpu(p: inputs.Problem, config=None, flags: int = 0) -> np.ndarray:
    A, W, R = (t.cuda() for t in (p.A, p.W, p.R))
    if config is None and flags == 0:
        Y = sgr.skinny_gemm_residual(A, W, R)
    else:
        Y = sgr.skinny_gemm_residual_ex(A, W, R, flags=flags, config=config)
    torch.cuda.synchronize()
    return bits(Y)


# ------------------------------------------------------------ small shapes
SMALL = [  # (M, N, K): several CTAs and ring stages plus ragged tails
    (1, 520, 264), (2, 1000, 1032), (3, 7168, 64), (4, 2056, 3584), (5, 304, 8),
    (7, 1512, 1800), (8, 4104, 3584), (11, 800, 7168), (16, 2056, 3584), (16, 8, 3584),
    (1, 8, 8), (13, 152, 1792),
]


@pytest.mark.parametrize("M,N,K", SMALL)
def test_parity_small_shapes(M, N, K):
    p = inputs.make_problem(M, N, K, seed=M * 1000 + N + K)
    compare(run_gpu(p), oracle_full(p.A, p.W, p.R), f"{M}x{N}x{K}")


# ------------------------------------------------------------ full sizes
@pytest.mark.parametrize("M", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_parity_full_size_every_element(M, seed):
    """The latent-MoE projection shape, M sweep x the four rotating seeds,
    every output element against the oracle."""
    p = inputs.make_problem(M, N_FULL, K_FULL, seed=seed)
    m = compare(run_gpu(p), oracle_full(p.A, p.W, p.R), f"M={M} seed={seed}")
    assert m["cosine"] > 0.999


# The down-projection of the same block (K = 7168 -> N = 3584): through the
# library's choice, the row slab with the 2-CTA K split (48-row slabs, one CTA
# per half of K) up to 64 tokens, each table entry and the M between them.
N_DOWN, K_DOWN = 3584, 7168


@pytest.mark.parametrize("M", [1, 2, 3, 4, 8, 16, 24, 32, 40, 48, 64, 100, 128])
def test_parity_down_projection_every_element(M):
    p = inputs.make_problem(M, N_DOWN, K_DOWN, seed=500 + M)
    m = compare(run_gpu(p), oracle_full(p.A, p.W, p.R), f"down M={M}")
    assert m["cosine"] > 0.999


@pytest.mark.parametrize("M", [256, 512, 1024])
def test_parity_down_projection_every_element_large_m(M):
    p = inputs.make_problem(M, N_DOWN, K_DOWN, seed=500 + M)
    m = compare(run_gpu(p), oracle_full(p.A, p.W, p.R), f"down M={M}")
    assert m["cosine"] > 0.999


@pytest.mark.parametrize("M", [256, 512, 1024])
def test_parity_compute_bound_sweep_every_element(M):
    """The compute-bound sweep at the latent-MoE shape through the library's
    own choice of kernel: every output element."""
    p, ref = oracle_problem(M, N_FULL, K_FULL, seed=M)
    m = compare(run_gpu(p), ref, f"M={M}")
    assert m["cosine"] > 0.999


@pytest.mark.parametrize("M", [32, 64, 128])
def test_parity_transition_sweep_every_element(M):
    """The transition sweep at the latent-MoE shape through the library's own
    choice of kernel: every output element."""
    p, ref = oracle_problem(M, N_FULL, K_FULL, seed=M + 1)
    m = compare(run_gpu(p), ref, f"M={M}")
    assert m["cosine"] > 0.999


@pytest.mark.parametrize("kb,stages", [(4, 4), (8, 3), (8, 2), (2, 6)])
@pytest.mark.parametrize("M", [1, 7, 16])
def test_parity_down_projection_rows_packing(kb, stages, M):
    """Row slab with 24 rows: 4 (kb = 4, 8) or 2 (kb = 2) K blocks per MMA,
    combined by the decode epilogue."""
    p = inputs.make_problem(M, N_DOWN, K_DOWN, seed=600 + M + kb)
    cfg = sgr.make_config(path=sgr.SGR_PATH_TC_ROWS, k_blocks_per_stage=kb, stages=stages)
    compare(run_gpu(p, config=cfg), oracle_full(p.A, p.W, p.R), f"down rows M={M} kb={kb}")


@pytest.mark.parametrize("M", [3, 5, 6, 7, 9, 12, 15])
def test_parity_full_size_odd_m(M):
    p = inputs.make_problem(M, N_FULL, K_FULL, seed=100 + M)
    compare(run_gpu(p), oracle_full(p.A, p.W, p.R), f"M={M}")


def test_parity_unit_normal_weights():
    """The vLLM benchmark page draws W ~ N(0,1) (no 1/sqrt(K) scale)."""
    p = inputs.make_problem(4, N_FULL, K_FULL, seed=5, w_scale=1.0)
    compare(run_gpu(p), oracle_full(p.A, p.W, p.R), "unit-normal W")


def test_integer_inputs_are_exact():
    """Integer inputs keep every FP32 partial sum exact, so any summation
    order gives the exact integer, and one rounding of it gives the
    oracle's bits."""
    M, N, K = 16, 2048, 512
    A = inputs.integer_bf16((M, K), -2, 2, 1)
    W = inputs.integer_bf16((N, K), -2, 2, 2)
    R = inputs.integer_bf16((M, N), -8, 8, 3)
    want = (A.to(torch.int64) @ W.to(torch.int64).T + R.to(torch.int64))
    assert want.abs().max() < 2 ** 24  # every FP32 partial sum is an exact integer
    Y = sgr.skinny_gemm_residual(A.cuda(), W.cuda(), R.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(bits(Y), bits(want.to(torch.bfloat16)))


# ------------------------------------------------------------ configurations
SIMT_CONFIGS = [
    dict(ctas_per_sm=1, rows_per_stage=1, stages=4),
    dict(ctas_per_sm=1, rows_per_stage=2, stages=12),
    dict(ctas_per_sm=2, rows_per_stage=2, stages=6),
    dict(ctas_per_sm=2, rows_per_stage=1, stages=8),
    dict(ctas_per_sm=1, rows_per_stage=4, stages=6),
    dict(ctas_per_sm=3, rows_per_stage=1, stages=4),
]


@pytest.mark.parametrize("cfg", SIMT_CONFIGS, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
@pytest.mark.parametrize("M", [1, 4, 16])
def test_parity_simt_configs(cfg, M):
    p = inputs.make_problem(M, N_FULL, K_FULL, seed=7)
    c = sgr.make_config(path=sgr.SGR_PATH_SIMT, **cfg)
    compare(run_gpu(p, config=c), oracle_full(p.A, p.W, p.R), f"M={M} {cfg}")


def test_unsupported_config_is_rejected_without_launch():
    p = inputs.make_problem(2, 520, 264, seed=1)
    A, W, R = (t.cuda() for t in (p.A, p.W, p.R))
    Y = torch.full_like(R, 7.0)
    c = sgr.make_config(path=sgr.SGR_PATH_SIMT, stages=64, rows_per_stage=64)
    with pytest.raises(sgr.SgrError) as e:
        sgr.skinny_gemm_residual_ex(A, W, R, Y, config=c)
    assert e.value.status == sgr.SGR_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(Y == 7.0)


# ------------------------------------------------------------ layouts
def test_strided_operands():
    """A, R, Y as column slices of wider buffers (row strides > row width)."""
    M, N, K = 4, 2048, 1024
    p = inputs.make_problem(M, N, K, seed=11)
    Abig = torch.zeros((M, K + 64), dtype=torch.bfloat16, device="cuda")
    Rbig = torch.zeros((M, 2 * N), dtype=torch.bfloat16, device="cuda")
    Ybig = torch.full((M, N + 512), 3.0, dtype=torch.bfloat16, device="cuda")
    A = Abig[:, 32:32 + K]
    A.copy_(p.A)
    R = Rbig[:, N:]
    R.copy_(p.R)
    Y = Ybig[:, 256:256 + N]
    sgr.skinny_gemm_residual_ex(A, p.W.cuda(), R, Y)
    torch.cuda.synchronize()
    compare(bits(Y), oracle_full(p.A, p.W, p.R), "strided")
    assert torch.all(Ybig[:, :256] == 3.0) and torch.all(Ybig[:, 256 + N:] == 3.0)


def test_in_place_residual():
    p = inputs.make_problem(8, N_FULL, K_FULL, seed=12)
    A, W = p.A.cuda(), p.W.cuda()
    RY = p.R.cuda().clone()
    sgr.skinny_gemm_residual(A, W, RY, RY)
    torch.cuda.synchronize()
    compare(bits(RY), oracle_full(p.A, p.W, p.R), "in-place")


def test_guard_bands_untouched():
    """Output written exactly inside [Y, Y + M*N): canaries around it survive."""
    M, N, K = 5, 1544, 512
    p = inputs.make_problem(M, N, K, seed=13)
    pad = 4096
    buf = torch.full((M * N + 2 * pad,), -5.0, dtype=torch.bfloat16, device="cuda")
    Y = buf[pad:pad + M * N].view(M, N)
    sgr.skinny_gemm_residual(p.A.cuda(), p.W.cuda(), p.R.cuda(), Y)
    torch.cuda.synchronize()
    assert torch.all(buf[:pad] == -5.0) and torch.all(buf[pad + M * N:] == -5.0)
    compare(bits(Y), oracle_full(p.A, p.W, p.R), "guarded")


# ------------------------------------------------------------ edge cases
def test_k_zero_copies_residual():
    M, N = 3, 64
    R = inputs.make_rows(M, N, 3).cuda()
    Y = torch.zeros_like(R)
    A = torch.empty((M, 0), dtype=torch.bfloat16, device="cuda")
    W = torch.empty((N, 0), dtype=torch.bfloat16, device="cuda")
    rc = sgr.skinny_gemm_residual_ex_ptr(A.data_ptr(), 0, W.data_ptr(), R.data_ptr(), N,
                                         Y.data_ptr(), N, M, N, 0, 0,
                                         torch.cuda.current_stream().cuda_stream)
    assert rc == sgr.SGR_OK
    torch.cuda.synchronize()
    assert torch.equal(Y, R)


def test_empty_m_is_a_no_op():
    W = inputs.make_weights(64, 64, 1).cuda()
    A = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    R = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    Y = sgr.skinny_gemm_residual(A, W, R)
    torch.cuda.synchronize()
    assert Y.shape == (0, 64)


def test_rejections_leave_output_untouched():
    M, N, K = 2, 256, 256
    p = inputs.make_problem(M, N, K, seed=2)
    A, W, R = (t.cuda() for t in (p.A, p.W, p.R))
    Y = torch.full_like(R, 9.0)
    s = torch.cuda.current_stream().cuda_stream
    # misaligned A (offset by one element), Y aliasing A, odd N
    Abuf = torch.zeros(M * K + 8, dtype=torch.bfloat16, device="cuda")
    assert sgr.skinny_gemm_residual_ptr(Abuf.data_ptr() + 2, W.data_ptr(), R.data_ptr(),
                                        Y.data_ptr(), M, N, K, s) == sgr.SGR_ERR_ALIGN
    assert sgr.skinny_gemm_residual_ptr(A.data_ptr(), W.data_ptr(), R.data_ptr(),
                                        A.data_ptr(), M, N, K, s) == sgr.SGR_ERR_ALIAS
    assert sgr.skinny_gemm_residual_ptr(A.data_ptr(), W.data_ptr(), R.data_ptr(),
                                        Y.data_ptr(), M, N - 4, K, s) == sgr.SGR_ERR_SHAPE
    torch.cuda.synchronize()
    assert torch.all(Y == 9.0)


# ------------------------------------------------------------ launch modes
def test_deterministic_and_pdl_independent():
    p = inputs.make_problem(4, N_FULL, K_FULL, seed=21)
    y1 = run_gpu(p)
    y2 = run_gpu(p)
    y3 = run_gpu(p, flags=sgr.SGR_FLAG_NO_PDL)
    assert np.array_equal(y1, y2) and np.array_equal(y1, y3)


def test_graph_capture_matches_eager():
    """Calls captured in a CUDA graph (the benchmark's method) give the eager bits."""
    M = 4
    probs = [inputs.make_problem(M, N_FULL, K_FULL, seed=s) for s in range(3)]
    dev = [[t.cuda() for t in (q.A, q.W, q.R)] for q in probs]
    outs = [torch.empty_like(d[2]) for d in dev]
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for (A, W, R), Y in zip(dev, outs):  # eager warm-up on the capture stream
            sgr.skinny_gemm_residual(A, W, R, Y)
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()
    eager = [bits(Y) for Y in outs]
    for Y in outs:
        Y.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for (A, W, R), Y in zip(dev, outs):
            sgr.skinny_gemm_residual(A, W, R, Y)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for e, Y, q in zip(eager, outs, probs):
        assert np.array_equal(e, bits(Y))
    compare(eager[0], oracle_full(probs[0].A, probs[0].W, probs[0].R), "graph")


def test_chain_of_eight_layers():
    """Eight projections in a row, Y_i[:, :K] (row stride N) feeding A_{i+1},
    each with its own W_i and R_i.  The oracle runs each layer on the GPU's
    own input for that layer, so errors do not compound."""
    M, L = 4, 8
    Ws = [inputs.make_weights(N_FULL, K_FULL, 1000 + i) for i in range(L)]
    Rs = [inputs.make_rows(M, N_FULL, 2000 + i) for i in range(L)]
    A0 = inputs.make_rows(M, K_FULL, 3000)
    dW = [w.cuda() for w in Ws]
    dR = [r.cuda() for r in Rs]
    Ys = [torch.empty((M, N_FULL), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    A = A0.cuda()
    for i in range(L):
        sgr.skinny_gemm_residual_ex(A, dW[i], dR[i], Ys[i])
        A = Ys[i][:, :K_FULL]
    torch.cuda.synchronize()
    a_in = A0
    for i in range(L):
        compare(bits(Ys[i]), oracle_full(a_in, Ws[i], Rs[i]), f"layer {i}")
        a_in = Ys[i][:, :K_FULL].cpu()
