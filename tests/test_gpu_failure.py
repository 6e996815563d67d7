"""Failure detection without a GPU fault: a bounded wait that runs out records
its code in the device error word, the host reads it, and the context stays
usable for the next call."""
import pytest
import torch

import skinny_bf16_gemm_residual_gb300 as sgr
from skinny_bf16_gemm_residual_gb300 import inputs
from parity import bits, compare, oracle_full

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    torch.cuda.set_device(0)
    sgr.sgr_init(0)
    yield


@pytest.mark.parametrize("limit_us", [50, 2000])
def test_timed_out_wait_is_reported_and_context_survives(limit_us):
    assert sgr.sgr_selftest_wait_timeout(limit_us) == 1  # a consumer gave up waiting
    assert sgr.sgr_device_error(0) == 0                  # the self-test cleared the word
    p = inputs.make_problem(4, 1024, 512, seed=11)
    Y = sgr.skinny_gemm_residual(p.A.cuda(), p.W.cuda(), p.R.cuda())
    torch.cuda.synchronize()
    compare(bits(Y), oracle_full(p.A, p.W, p.R), "call after a timed-out wait")
    assert sgr.sgr_device_error(0) == 0


def test_selftest_rejects_bad_limits():
    for bad in (0, 100001):
        with pytest.raises(sgr.SgrError) as e:
            sgr.sgr_selftest_wait_timeout(bad)
        assert e.value.status == sgr.SGR_ERR_UNSUPPORTED


@pytest.mark.parametrize("M,N,K,cta", [(16, 7168, 3584, 0), (16, 7168, 3584, 75), (16, 7168, 3584, 151),
                                       (4, 1024, 2048, 3), (40, 2048, 1024, 1)])
def test_streamk_abort_leaves_counters_clean(M, N, K, cta):
    """A stream-K CTA that gives up waiting still arrives on the split-K tile
    counters: the next stream-K call on the same tiles must match the oracle
    (a counter left short would make an early arriver sum missing partials)."""
    p = inputs.make_problem(M, N, K, seed=40 + cta)
    A, W, R = (t.cuda() for t in (p.A, p.W, p.R))
    c = sgr.sgr_default_config(M, N, K, sgr.SGR_PATH_TC)
    import math
    grid = min(torch.cuda.get_device_properties(0).multi_processor_count * c.ctas_per_sm,
               math.ceil(N / 128) * math.ceil(M / c.token_tile) * math.ceil(K / (64 * c.k_blocks_per_stage)))
    cta = min(cta, grid - 1)
    Y = torch.empty_like(R)
    assert sgr.sgr_selftest_streamk_abort(A, W, R, Y, cta) == 3  # the epilogue gave up waiting
    assert sgr.sgr_device_error(0) == 0                          # the self-test cleared the word
    ref = oracle_full(p.A, p.W, p.R)
    for _ in range(2):
        y = sgr.skinny_gemm_residual_config(A, W, R, config=sgr.make_config(path=sgr.SGR_PATH_TC))
        torch.cuda.synchronize()
        compare(bits(y), ref, f"stream-K call after an aborted CTA {cta} (M={M} N={N} K={K})")
    assert sgr.sgr_device_error(0) == 0


def test_streamk_abort_rejects_bad_cta():
    p = inputs.make_problem(4, 1024, 512, seed=12)
    A, W, R = (t.cuda() for t in (p.A, p.W, p.R))
    for bad in (-1, 1 << 20):
        with pytest.raises(sgr.SgrError) as e:
            sgr.sgr_selftest_streamk_abort(A, W, R, torch.empty_like(R), bad)
        assert e.value.status == sgr.SGR_ERR_UNSUPPORTED
