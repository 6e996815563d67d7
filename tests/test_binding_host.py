"""Host-side checks of the Python binding that need no GPU: tensor dtype,
rank and inner-stride rules, one device for every operand, and a stream on
that device.  Stand-in objects carry only the attributes the checks read."""
import pytest
import torch

from skinny_bf16_gemm_residual_gb300 import binding


class FakeCuda:
    """A 2-D CUDA tensor as far as the binding's checks can tell."""

    def __init__(self, shape, strides, device="cuda:0", dtype=torch.bfloat16):
        self.shape, self._strides = tuple(shape), tuple(strides)
        self.device, self.dtype, self.is_cuda = torch.device(device), dtype, True

    def dim(self):
        return len(self.shape)

    def stride(self, i):
        return self._strides[i]


class FakeStream:
    def __init__(self, device):
        self.device, self.cuda_stream = torch.device(device), 1234


def test_check_tensor_accepts_row_strided_views():
    binding._check_tensor(FakeCuda((4, 3584), (3600, 1)), "A")
    binding._check_tensor(FakeCuda((1, 3584), (3584, 1)), "A")
    binding._check_tensor(FakeCuda((1, 3584), (1, 1)), "A")  # one row: its row stride is never used


@pytest.mark.parametrize("t,err", [
    (FakeCuda((4, 3584), (3584, 2)), ValueError),           # every other column
    (FakeCuda((1, 3584), (7168, 2)), ValueError),           # one row, still strided columns
    (FakeCuda((3584, 4), (1, 3584)), ValueError),           # a transposed view
    (FakeCuda((4, 3584), (3584, 1), dtype=torch.float16), TypeError),
    (FakeCuda((4, 3584, 1), (3584, 1, 1)), ValueError),
])
def test_check_tensor_rejects(t, err):
    with pytest.raises(err):
        binding._check_tensor(t, "A")


def test_check_tensor_rejects_host_tensors():
    with pytest.raises(ValueError):
        binding._check_tensor(torch.zeros((2, 8), dtype=torch.bfloat16), "A")


def test_operands_on_one_device():
    a, b = FakeCuda((1, 8), (8, 1), "cuda:1"), FakeCuda((8, 8), (8, 1), "cuda:1")
    assert binding._common_device((a, b)) == torch.device("cuda:1")
    with pytest.raises(ValueError, match="one CUDA device"):
        binding._common_device((a, FakeCuda((8, 8), (8, 1), "cuda:0")))


def test_stream_on_the_operands_device():
    dev = torch.device("cuda:1")
    assert binding._stream_handle(FakeStream("cuda:1"), dev) == 1234
    assert binding._stream_handle(77, dev) == 77  # a raw handle is taken as given
    with pytest.raises(ValueError, match="stream is on"):
        binding._stream_handle(FakeStream("cuda:0"), dev)
