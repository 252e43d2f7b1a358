"""Testing the instrument: planted-fault builds of the oracle must fail at
least one pin each ("The kernel reference interpreter", section "Testing the
instrument": a known-wrong variant exists only so that a test can show it is
caught).  Faults are planted in the oracle, on the CPU, never in GPU code."""
import pytest

import oracle
import pins

FAULTS = {
    1: "min term dropped",
    2: "Q4_K nibble halves swapped",
    3: "Q4_K upper scales and mins swapped",
    4: "codebook nibble halves swapped",
    5: "q8 ties rounded away from zero",
    6: "q8 sub-block sums in the wrong slot",
    7: "min term sign flipped",
    8: "q8 scale step amax/128",
    9: "RMSNorm eps dropped",
    10: "RMSNorm wave lanes added left to right",
    11: "RMSNorm item loop reversed",
    12: "resident payload written without the prefix offset",
    13: "resident scale bytes swapped",
}


@pytest.mark.parametrize("fault", sorted(FAULTS), ids=lambda f: FAULTS[f])
def test_planted_fault_is_caught(fault):
    o = oracle.Oracle(fault)
    failed = []
    for pin in pins.ALL_PINS:
        if pin is pins.pin_f16_all_patterns:
            continue
        try:
            pin(o)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"planted fault {fault} ({FAULTS[fault]}) passed every pin"
