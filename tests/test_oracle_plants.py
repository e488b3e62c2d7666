"""Each deliberate mistake compiled into the oracle must make at least one pin fail.

The plants (sites marked PLANT(n) in oracle/moe_oracle.cpp) are the kinds of
error the pins are meant to catch: a dropped bias term, a wrong tie-break, a
transposed operand, a capacity formula without k, a wrong GELU or SiLU, missing
renormalisation, reversed dropping order, a missing factor in the aux loss and
an unsquared z-loss, a pass-through of tokens that kept an expert, a shard
that ignores the earlier shards' counts, and three MXFP8 slips (scale exponent,
tie rule, a skipped quantisation). Only the oracle is planted, on the CPU.
"""
import os

import pytest

import oracle
import oracle_pins

PLANTS = {
    1: "GELU expert without its first bias",
    2: "top-k ties go to the higher index",
    3: "W2 indexed as [F, d] instead of [d, F]",
    4: "capacity without the factor k",
    5: "GELU without the 1/sqrt(2)",
    6: "SiLU with the wrong sign",
    7: "renormalised gates not renormalised",
    8: "dropping keeps the last C tokens",
    9: "aux loss without the factor E",
    10: "z-loss not squared",
    11: "pass-through for a token with any dropped slot",
    12: "shard ranks without the earlier shards' counts",
    13: "MX shared exponent one too small (floor(log2 max) - 7)",
    14: "E4M3 rounding ties away from zero",
    15: "MXFP8 experts without the hidden-row quantisation",
}


@pytest.mark.parametrize("plant", sorted(PLANTS), ids=lambda n: PLANTS[n])
def test_plant_is_caught(plant, tmp_path):
    path = oracle.build(out_path=os.path.join(tmp_path, f"liboracle_plant{plant}.so"), plant=plant)
    o = oracle.Oracle(path)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught plant {plant}: {PLANTS[plant]}"
