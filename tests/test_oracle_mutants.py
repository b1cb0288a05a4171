"""Mutant check of the oracle pins.

Each planted mistake is compiled into a separate build of the oracle
(``-DORACLE_MUTANT=n``, CPU only) and must fail at least one pin.  The list
follows the pitfalls table of "FlashAttention forward in C" (section 5) where
a pitfall applies to a plain, untiled definition (s03-s09, s15), plus generic
slips: a dropped scale, a scaled mask, a transposed operand, a flipped sign,
swapped mask strides, a scaled sink and a missing max subtraction.  s01, s02,
s10-s14 concern tiles, arenas and threads; the GPU invariance tests cover the
tiled kernels.
"""
from pathlib import Path

import pytest

import oracle
from oracle_pins import ALL_PINS

MUTANTS = {
    3: "round-robin KV head map (h mod Hkv)",
    4: "causal as j < p",
    5: "window of w + 1 keys",
    6: "q_offset ignored",
    7: "sink left out of the denominator",
    8: "lse without the maximum",
    9: "empty row divides by zero",
    15: "H mod Hkv != 0 accepted",
    20: "scale dropped",
    21: "mask scaled with the dot product",
    22: "keys used as values",
    23: "exponent sign flipped",
    24: "mask strides swapped",
    25: "sink logit scaled",
    26: "maximum not subtracted",
}

_DIR = Path(oracle.__file__).resolve().parent / "_mutants"


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=[f"m{m}" for m in sorted(MUTANTS)])
def test_mutant_is_caught(mutant):
    lib = oracle.build(mutant=mutant, out=_DIR / f"libfa_oracle_m{mutant}.so")
    orc = oracle.Oracle(lib)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {mutant} ({MUTANTS[mutant]}) passed every pin"
