"""Planted mistakes in the oracle must each fail at least one pin.

Each mutant is the oracle's C source rebuilt with -DORACLE_MUTANT=<n>, which
swaps one line for a plausible mistake (a dropped term, an inverted ratio, a
wrong sign, a missing square root, a boundary that clips ...).  A pin suite
that lets one of them through is too weak to trust the oracle with.
"""
import pytest

import oracle
from _pins import ALL_PINS

MUTANTS = {
    1: "unscale dropped from the sum of squares",
    2: "unscale applied twice in the sum of squares",
    3: "L1 instead of L2",
    4: "last element of each tensor dropped",
    5: "only the first tensor counted",
    6: "norm == max_norm clips",
    7: "ratio inverted (norm / max_norm)",
    8: "square root missing",
    9: "outputs not unscaled",
    10: "sign of the output flipped",
    11: "AdamW without bias correction",
    12: "AdamW eps inside the square root",
    13: "AdamW weight decay coupled into the gradient",
    14: "AdamW fed the unclipped gradient",
    15: "AdamW second moment with beta1",
    16: "accumulation subtracts the last microbatch",
    17: "each contribution clipped before it is added",
    18: "per-tensor clipping applies the global clip",
    19: "the fp32 output loses the clip factor",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: f"m{m}")
def test_mutant_is_caught(mutant, tmp_path_factory):
    o = oracle.Oracle(mutant, str(tmp_path_factory.mktemp(f"mutant{mutant}")))
    caught = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {mutant} ({MUTANTS[mutant]}) passed every pin"
