"""Plant one plausible mistake at a time in the oracle (on the CPU: oracle.c
built with -DORACLE_MUTANT=n) and require that at least one pin rejects
each copy.  This is what makes the pins worth trusting: a dropped term, a
wrong sign, constant or index, a transposed operand or a double rounding
anywhere in the oracle shows up as a failing pin."""
import pytest

import oracle
from tests import pins

MUTANTS = {
    1: "encode: ties away from zero",
    2: "decode: wrong subnormal exponent",
    3: "scale: another format's maximum (240)",
    4: "gemm: last K block dropped",
    5: "gemm: weight scales read transposed",
    6: "gemm: activation scales read transposed",
    7: "bf16 rounding through fp32 first",
    8: "weight amax: signed maximum",
    9: "gemm: weight operand read transposed",
    10: "encode: sign of zero dropped",
    11: "encode: overflow to NaN instead of saturating",
    12: "greedy: ties to the highest column",
    13: "greedy: -0 ranked below +0",
    14: "MX: another element maximum exponent (7)",
    15: "MX: ceiling instead of floor of log2(amax)",
}


@pytest.mark.parametrize("n", sorted(MUTANTS), ids=lambda n: "mutant%d" % n)
def test_some_pin_rejects_mutant(n):
    m = oracle.mutant(n)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(m)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, "no pin catches: " + MUTANTS[n]
