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
