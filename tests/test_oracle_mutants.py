"""Pin sensitivity: the oracle rebuilt with one planted mistake at a time
(-DOR_MUTANT=n, see the header of oracle/bpkv_oracle.c) must fail at least one
pin.  The mistakes are plausible slips in reading the Fathom page: bit or plane
order, floor vs round, the mid-rise half step, the scale's cost, q^2 vs |q|,
tie rules, the 1/sqrt(D) factor, the union mask, stop vs skip, the
calibration statistic, the basis orientation, and in the ReadKV page's
value stage the weight (squared probabilities), its tie rule and the
channel order of a value plane."""
import pytest

from pins import ALL_PINS

MUTANTS = {
    1: "token-to-bit order reversed inside a plane word",
    2: "plane 0 holds the least significant code bit",
    3: "dequantisation without the half step (mid-tread)",
    4: "first bit of a channel costs no scale",
    5: "top-k ties go to the higher index",
    6: "importance uses |q| instead of q^2",
    7: "code rounds k/s to nearest instead of floor",
    8: "attention logits miss 1/sqrt(D)",
    9: "union mask keeps only the first head",
    10: "allocator skips an unaffordable item instead of stopping",
    11: "calibrated channel sets rank by mean |q| alone",
    12: "calibrated channel sets average q^2 instead of |q|",
    13: "basis applied transposed",
    14: "value-row weights sum the attention probabilities, not their squares",
    15: "value-depth ties go to the higher row",
    16: "value planes hold the channels of a word in reverse order",
}


@pytest.mark.parametrize("n", sorted(MUTANTS), ids=[MUTANTS[k] for k in sorted(MUTANTS)])
def test_mutant_is_caught(n):
    from oracle import load_variant
    o = load_variant([f"-DOR_MUTANT={n}"])
    failed = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin catches mutant {n}: {MUTANTS[n]}"
