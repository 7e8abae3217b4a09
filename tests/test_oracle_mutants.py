"""Plant one mistake at a time in the CPU oracle and check that a pin catches it.

The oracle is recompiled with -DORC_MUTANT=n (a dropped term, a wrong order, a transposed
operand, a missing step ...) into a scratch directory; the pin that guards that step must
fail against the mutant.  CPU only; the trusted oracle (ORC_MUTANT=0) is restored afterwards.
"""
import os
import subprocess

import pytest

from oracle import oracle as O

from . import test_oracle_pins as pins

MUTANTS = {
    1: ("int4 nibble order swapped", ["test_int4_nibble_exhaustive"]),
    2: ("q8 truncates instead of rounding", ["test_q8_golden"]),
    3: ("exp polynomial drops its r^4 term", ["test_exp_within_two_ulp"]),
    4: ("SwiGLU applies SiLU to u instead of g", ["test_expert_ffn_against_fp64"]),
    5: ("canonical dot uses strided groups", ["test_canon_dot_groups_are_contiguous"]),
    6: ("top-k ties go to the higher index", ["test_topk_equals_full_stable_sort"]),
    7: ("routing weights from biased scores", ["test_router_bias_changes_selection_not_weights"]),
    8: ("combine drops the shared expert", ["test_forced_all_experts_equals_dense_loop"]),
    9: ("residual add missing after RMSNorm", ["test_norm_layer_is_residual_of_plain_layer"]),
    10: ("RMSNorm without eps", ["test_rmsnorm_closed_form"]),
    11: ("bucket records the wrong rank", ["test_union_bucket_brute_force"]),
    12: ("block dot pairs block b with block nb-1-b", ["test_matvec_accumulators_brute_force"]),
    13: ("int8 row codes clamped to 126", ["test_int8_row_quant_bounds", "test_int8_row_quant_golden",
                                            "test_int8_codes_round_trip_exhaustively"]),
    14: ("int8 block dot drops the block's last element", ["test_i8_block_dot_brute_force",
                                                           "test_i8_matvec_accumulators_brute_force"]),
    15: ("int2 fields read from the high bits down", ["test_int2_decode_golden", "test_int2_pack_exhaustive",
                                                       "test_i2_block_dot_brute_force"]),
    16: ("int2 codes not sign-extended", ["test_int2_decode_golden", "test_int2_pack_exhaustive",
                                          "test_i2_matvec_accumulators_brute_force"]),
    17: ("int2 row scale max|w|/2", ["test_int2_row_quant_golden", "test_int2_row_quant_bounds"]),
    18: ("int8 expert records read at the int4 offsets", ["test_expert_of_equal_codes_is_the_same_in_every_width",
                                                          "test_int8_expert_against_fp64",
                                                          "test_layer_of_equal_codes_is_the_same_in_every_width"]),
    19: ("fp64 layer output reads down rows at the int4 offset", [
        "test_layer_of_equal_codes_is_the_same_in_every_width"]),
}


@pytest.fixture
def mutant_lib(tmp_path):
    saved_so, saved_lib = O.SO, O._lib

    def use(n):
        so = str(tmp_path / f"liboracle_m{n}.so")
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off",
                               f"-DORC_MUTANT={n}", os.path.join(O.HERE, "oracle.c"), "-o", so,
                               "-lm"])
        O.SO, O._lib = so, None
        O.lib()

    yield use
    O.SO, O._lib = saved_so, saved_lib


@pytest.mark.parametrize("n", sorted(MUTANTS))
def test_pin_catches_planted_mistake(n, mutant_lib):
    what, guards = MUTANTS[n]
    mutant_lib(n)
    for name in guards:
        with pytest.raises(AssertionError):
            getattr(pins, name)()
