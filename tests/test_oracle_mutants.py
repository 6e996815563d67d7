"""Each planted mistake in the oracle must be caught by at least one pin.

The mistakes are compiled into separate copies of the oracle (CPU only):
1 residual dropped, 2 product rounded before the residual add, 3 last k
dropped, 4 residual subtracted, 5 truncation instead of nearest-even,
6 ties away from zero, 7 FP32 running sum, 8 residual read from the wrong row;
in the low-bit weight variant: 9 E4M3 subnormals decoded as normals, 10 E4M3
exponent bias 8, 11 residual multiplied by the scale, 12 no NaN code (0x7F
read as 480), 13 the scale of the neighbouring column; in the NVFP4 variant:
14 nibble order swapped, 15 one block scale per 32 elements instead of 16,
16 E2M1 subnormals decoded as normals, 17 residual multiplied by the tensor
scale.
"""
import pytest

import oracle
import pins


@pytest.mark.parametrize("mutant", range(1, 18))
def test_planted_mistake_is_caught(tmp_path_factory, mutant):
    lib = oracle.load(mutant, out_dir=str(tmp_path_factory.getbasetemp() / "mutants"))
    assert lib.mutant == mutant
    failed = []
    for check in pins.ALL_CHECKS:
        try:
            check(lib)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"mutant {mutant} passed every pin"
