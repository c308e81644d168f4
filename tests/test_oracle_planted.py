"""The pins catch plausible mistakes (no GPU).

Each case compiles the oracle with one deliberate mistake (the ORC_PLANT list
in oracle/oracle.c) into a separate library and runs, against it, the pins
that should expose it: at least one of them must fail.  The regular library
is restored afterwards, and every pin passes on it (the other test files)."""
import pytest

import test_oracle_fos as fos
import test_oracle_formats as fmt
import test_oracle_layer as lay
import test_oracle_mxfp8 as mx
import test_oracle_routing as rt

CASES = [
    (1, "softmax scores replaced by sigmoid",
     [rt.test_softmax_two_experts_is_the_logistic_of_the_difference,
      rt.test_softmax_is_shift_invariant_and_sigmoid_is_not]),
    (2, "normalisation ignored",
     [rt.test_scores_weights_closed_form, rt.test_weights_sum_to_one_and_permutation]),
    (3, "gate and up rows swapped",
     [lay.test_closed_form_tiny_layer, lay.test_closed_form_two_experts_and_shared]),
    (4, "shared experts dropped from the combine",
     [lay.test_shared_expert_only, lay.test_closed_form_two_experts_and_shared]),
    (5, "E2M1 subnormal decoded as 1.0",
     [fmt.test_e2m1_golden_file, fmt.test_e2m1_table_exhaustive]),
    (6, "MX scales taken per 16 elements instead of per 32",
     [lambda orc: mx.test_dequant_matches_nvfp4_on_shared_values(orc, "mxfp4"),
      lambda orc: mx.test_layer_matches_nvfp4_on_shared_values(orc, "mxfp8", "mxfp8")]),
    (7, "FP8 block scales indexed with rows and columns swapped",
     [lambda orc: mx.test_dequant_matches_nvfp4_on_shared_values(orc, "fp8_block"),
      mx.test_fp8_block_single_expert_equals_dense_mlp]),
    (8, "Four-Over-Six keeping the candidate with the larger error",
     [fos.test_four_wins_where_it_is_exact, fos.test_six_wins_where_it_is_exact]),
    (9, "Four-Over-Six ties going to 4",
     [fos.test_tie_goes_to_six_and_zero_rows]),
]


@pytest.mark.parametrize("plant,what,pins", CASES, ids=[c[1] for c in CASES])
def test_planted_mistake_is_caught(orc, plant, what, pins):
    caught = []
    with orc.planted(plant):
        for pin in pins:
            try:
                pin(orc)
            except AssertionError:
                caught.append(getattr(pin, "__name__", "pin"))
    assert caught, f"no pin caught the planted mistake: {what}"
    # and the regular oracle is back
    assert orc.e2m1(1) == 0.5
