"""The stored page values under tests/golden/ and how the tests read them."""
import math

from parity import TIGHT_ATOL, TIGHT_FRAC, TIGHT_MAX, TIGHT_RTOL, load_gate


def test_fp16_gate_fixture_complete():
    gate = load_gate()
    assert set(gate) == {"atol", "rtol", "max_abs_limit", "required_ratio"}
    assert TIGHT_FRAC == gate["required_ratio"] == 0.99
    assert TIGHT_MAX == gate["max_abs_limit"] == 0.1


def test_fp16_gate_tolerances_are_the_printed_powers_of_two():
    # the printed three-figure values round the powers of two the gate uses
    gate = load_gate()
    for printed, used, exp in ((gate["atol"], TIGHT_ATOL, -14), (gate["rtol"], TIGHT_RTOL, -9)):
        assert used == 2.0 ** exp
        digits = -math.floor(math.log10(printed)) + 2       # three significant figures
        assert round(used, digits) == printed
