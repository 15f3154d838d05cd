"""Mutation self-check of the pins (CPU only).

Each planted mistake is compiled into a separate build of the oracle; the pin
suite must reject every one of them.  The mistakes are the ones the pages warn
about (the two wrong head maps of the kv-copies-gqa head-map table) plus the
plausible slips in each step: an off-by-one or top-left causal mask, a
dropped log-sum in the LSE, a dropped softmax scale, page and slot swapped,
an ungated (identity) gate, the wrong FP8 exponent bias, a dropped v_scale,
and for whole-request paged decode an ignored sequence length, swapped
K / V scales or int8 codes read as unsigned.
"""
import os

import pytest

import oracle
from oracle_pins import ALL_PINS

MUTANTS = {
    1: "kv head (h // Hkv) % Hkv",
    2: "kv head h % Hkv",
    3: "causal mask off by one",
    4: "LSE = max score (log-sum dropped)",
    5: "softmax scale dropped",
    6: "page index and slot swapped",
    7: "gate applied without sigmoid",
    8: "E4M3 exponent bias 8",
    9: "v_scale dropped",
    10: "top-left causal alignment",
    11: "paged: per-request sequence length ignored",
    12: "paged: k_scale and v_scale swapped",
    13: "paged: int8 codes read as unsigned",
    14: "Dqk != Dv: scores summed over the value head size",
}


@pytest.mark.parametrize("bug", sorted(MUTANTS), ids=lambda b: f"bug{b}")
def test_pins_catch_mutant(tmp_path, bug):
    lib = oracle.build(out=os.path.join(str(tmp_path), f"liboracle_bug{bug}.so"), plant_bug=bug, force=True)
    orc = oracle.load(lib)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught planted bug {bug}: {MUTANTS[bug]}"
