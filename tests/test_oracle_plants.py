"""Mutation check of the pins: copies of the oracle compiled with one
plausible mistake each (wrong E2M1 bias, lost sign, wrong E8M0 bias,
swapped nibble order, column-major scale index, dropped last term, and in
the quantiser a wrong shared exponent, swapped nibbles, ties rounded up) must
each fail at least one pin.  The mistakes are planted in the oracle, on
the CPU, through compile-time macros of a separate build."""
import pytest

import oracle
import oracle_pins

PLANTS = ["OR_PLANT_E2M1_BIAS0", "OR_PLANT_E2M1_NOSIGN", "OR_PLANT_E8M0_BIAS128",
          "OR_PLANT_NIBBLE_SWAP", "OR_PLANT_SCALE_COLMAJOR", "OR_PLANT_DROP_LAST",
          # the quantiser: shared exponent one too high, codes in the wrong
          # nibbles, ties rounded up instead of to even
          "OR_PLANT_Q_EMAX", "OR_PLANT_Q_NIBBLE_SWAP", "OR_PLANT_Q_TIES_UP"]


@pytest.mark.parametrize("plant", PLANTS)
def test_pins_catch_planted_mistake(plant):
    planted = oracle.Oracle(defines=(plant,))
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(planted)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught {plant}"
