"""Plant a plausible mistake in the oracle (a rebuild of oracle.c with one ORC_PLANT_* macro)
and check that the pins catch it: each planted build must fail at least one pin."""
import pytest

import oracle
import oracle_pins as P

PLANTS = {
    "ORC_PLANT_EXP_TERM": "wrong Taylor coefficient in exp",
    "ORC_PLANT_ROUND_EVEN": "q8_1 codes rounded half to even",
    "ORC_PLANT_S_FROM_D16": "q8_1 s taken from the fp16 d",
    "ORC_PLANT_NIBBLE_ORDER": "4-bit codes read interleaved",
    "ORC_PLANT_SUB_NIBBLE": "CB sub-scale nibbles swapped",
    "ORC_PLANT_LS": "CB sub-scale used as sub instead of 2*sub+1",
    "ORC_PLANT_SIGN_ORDER": "CB sign bits read from the top",
    "ORC_PLANT_Q4B_MIN": "Q4B minimum term dropped",
    "ORC_PLANT_ROUTE_ORDER": "entries of a group ordered by slot first",
    "ORC_PLANT_ENTRY_ROW": "gate/up reads the entry index instead of its token row",
    "ORC_PLANT_SLOT_ORDER": "4-bit slot codes read interleaved",
    "ORC_PLANT_TIE_HIGH": "router ties resolved to the higher expert id",
    "ORC_PLANT_SOFTMAX_ALL": "router softmax over every expert instead of the selected k",
    "ORC_PLANT_COMBINE_SLOT": "combine drops the last slot",
    "ORC_PLANT_QSA_LANE_INTERLEAVE": "QSA lane slices strided (l, l+32, ...) instead of 4 consecutive dims",
    "ORC_PLANT_QSA_NO_FMA": "QSA lane products rounded before they are added",
    "ORC_PLANT_QSA_TREE_SEQ": "QSA lane partials summed in lane order instead of the warp-sum pairings",
    "ORC_PLANT_QSA_HEAD_ORDER": "QSA head relus summed in reverse order",
    "ORC_PLANT_QSA_TAIL_FIRST": "QSA +1e9 on the first block instead of the tail",
}


@pytest.mark.parametrize("plant", sorted(PLANTS))
def test_pins_catch_planted_mistake(plant):
    o = oracle.Oracle(defines=(plant,))
    failed = []
    for check in P.ALL_CHECKS:
        try:
            check(o)
        except AssertionError:
            failed.append(check.__name__)
            break
    assert failed, f"no pin caught: {PLANTS[plant]}"
