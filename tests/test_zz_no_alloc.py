"""The allocation-free entry point (skinny_gemm_residual_noalloc).

Some callers cannot allocate device memory at all: code running inside a
stream capture that forbids cudaMalloc, engines that reserve the whole
device memory up front, latency-critical paths that cannot afford the
synchronisation an allocation may imply.  The library therefore offers one
entry point whose split-K scratch lives in a fixed array inside the library.
This file checks, through the C ABI, that two calls in a row give the same
results as the regular entry point (within the parity tolerance), that the
scratch keeps working across calls, and that shapes beyond the fixed limit
are refused.  It is named so that pytest collects it last.
"""
from __future__ import annotations

import pytest
import torch

import skinny_bf16_gemm_residual_gb300 as sgr
from skinny_bf16_gemm_residual_gb300 import inputs
from parity import bits, compare

pytestmark = pytest.mark.gpu

N, K = inputs.N_LATENT_MOE, inputs.K_LATENT_MOE


def _noalloc(A, W, R, Y, stream):
    return sgr.skinny_gemm_residual_noalloc_ptr(
        A.data_ptr(), A.stride(0) if A.shape[0] > 1 else A.shape[1], W.data_ptr(), R.data_ptr(),
        R.stride(0) if R.shape[0] > 1 else R.shape[1], Y.data_ptr(),
        Y.stride(0) if Y.shape[0] > 1 else Y.shape[1], A.shape[0], W.shape[0], A.shape[1], 0, stream)


def test_noalloc_two_calls_match_regular_entry_point():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream().cuda_stream
    probs = [inputs.make_problem(4, N, K, seed=901), inputs.make_problem(16, N, K, seed=902)]
    dev = [[t.cuda() for t in (p.A, p.W, p.R)] for p in probs]
    outs = [torch.full_like(d[2], float("nan")) for d in dev]
    # Two allocation-free calls back to back on one stream, sharing the scratch,
    # made before anything else in this process touches the library's workspace.
    for (A, W, R), Y in zip(dev, outs):
        assert _noalloc(A, W, R, Y, stream) == sgr.SGR_OK
    torch.cuda.synchronize()
    for (A, W, R), Y, p in zip(dev, outs, probs):
        ref = sgr.skinny_gemm_residual(A, W, R)  # the regular entry point
        torch.cuda.synchronize()
        compare(bits(Y), bits(ref), f"noalloc M={p.M}")
    assert sgr.sgr_device_error(0) == 0


def test_noalloc_refuses_shapes_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    torch.cuda.set_device(0)
    p = inputs.make_problem(64, N, K, seed=903)
    A, W, R = (t.cuda() for t in (p.A, p.W, p.R))
    Y = torch.full_like(R, 5.0)
    rc = _noalloc(A, W, R, Y, torch.cuda.current_stream().cuda_stream)
    assert rc == sgr.SGR_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(Y == 5.0)
