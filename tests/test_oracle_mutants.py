"""Plant one mistake at a time in the CPU oracle and check that a pin catches it.

Each planted mistake (a dropped term, a wrong order, a transposed operand, a missing step ...)
is a text patch: `mutant_source(n)` applies it to a copy of oracle.c, which is compiled into a
scratch directory; the pin that guards that step must fail against the mutant.  The trusted
oracle.c carries no trace of the mistakes.  CPU only; the trusted library is restored
afterwards.
"""
import os
import subprocess

import pytest

from oracle import oracle as O

from . import test_oracle_pins as pins

# n: (what the mistake is, the pins that must catch it, [(trusted text, planted text), ...]).
# Each trusted text occurs exactly once in oracle.c.
MUTANTS = {
    1: ("int4 nibble order swapped", ["test_int4_nibble_exhaustive"],
        [("int nib = (j & 1) ? (byte >> 4) : (byte & 15);",
          "int nib = (j & 1) ? (byte & 15) : (byte >> 4);")]),
    2: ("q8 truncates instead of rounding", ["test_q8_golden"],
        [("v = (int)roundf(xb[j] / db);", "v = (int)truncf(xb[j] / db);")]),
    3: ("exp polynomial drops its r^4 term", ["test_exp_within_two_ulp"],
        [("p = fmaf(p, r, 0x1.555556p-5f); /* 1/4! */", "/* 1/4! dropped */")]),
    4: ("SwiGLU applies SiLU to u instead of g", ["test_expert_ffn_against_fp64"],
        [("float s = g / (1.0f + orc_exp(-g));\n  return s * u;",
          "float s = u / (1.0f + orc_exp(-u));\n  return s * g;")]),
    5: ("canonical dot uses strided groups", ["test_canon_dot_groups_are_contiguous"],
        [("      p[g] = fmaf(a[j], b[j], p[g]);",
          "      int jj = (j - g * G) * 32 + g;\n      if (jj < n) p[g] = fmaf(a[jj], b[jj], p[g]);")]),
    6: ("top-k ties go to the higher index", ["test_topk_equals_full_stable_sort"],
        [("if (best < 0 || sel[e] > sel[best])", "if (best < 0 || sel[e] >= sel[best])")]),
    7: ("routing weights from biased scores", ["test_router_bias_changes_selection_not_weights"],
        [("  float S = scores[ids[0]];\n  for (int k = 1; k < K; ++k) S = S + scores[ids[k]];",
          "  float S = sel[ids[0]];\n  for (int k = 1; k < K; ++k) S = S + sel[ids[k]];"),
         ("w[k] = (scores[ids[k]] / S) * routed_scale;", "w[k] = (sel[ids[k]] / S) * routed_scale;")]),
    8: ("combine drops the shared expert", ["test_forced_all_experts_equals_dense_loop"],
        [("float acc = ps >= 0 ? e[(int64_t)ps * d + r] : 0.0f;", "float acc = 0.0f;")]),
    9: ("residual add missing after RMSNorm", ["test_norm_layer_is_residual_of_plain_layer"],
        [("if (c->has_norm) acc = x[(int64_t)t * d + r] + acc;", "/* residual dropped */")]),
    10: ("RMSNorm without eps", ["test_rmsnorm_closed_form"],
         [("float r = 1.0f / sqrtf(ms + eps);", "float r = 1.0f / sqrtf(ms);")]),
    11: ("bucket records the wrong rank", ["test_union_bucket_brute_force"],
         [("pair_rank[p] = k;", "pair_rank[p] = K - 1 - k;")]),
    12: ("block dot pairs block b with block nb-1-b", ["test_matvec_accumulators_brute_force"],
         [("Ar[b] = orc_block_dot(wrow, qx, b);", "Ar[b] = orc_block_dot(wrow, qx, nb - 1 - b);")]),
    13: ("int8 row codes clamped to 126", ["test_int8_row_quant_bounds", "test_int8_row_quant_golden",
                                            "test_int8_codes_round_trip_exhaustively"],
         [("const int lim = 127;", "const int lim = 126;")]),
    14: ("int8 block dot drops the block's last element", ["test_i8_block_dot_brute_force",
                                                           "test_i8_matvec_accumulators_brute_force"],
         [("const int end = (b + 1) * QB;", "const int end = (b + 1) * QB - 1;")]),
    15: ("int2 fields read from the high bits down", ["test_int2_decode_golden", "test_int2_pack_exhaustive",
                                                       "test_i2_block_dot_brute_force"],
         [("const int k = j & 3;", "const int k = 3 - (j & 3);")]),
    16: ("int2 codes not sign-extended", ["test_int2_decode_golden", "test_int2_pack_exhaustive",
                                          "test_i2_matvec_accumulators_brute_force"],
         [("return code >= 2 ? code - 4 : code;", "return code;")]),
    17: ("int2 row scale max|w|/2", ["test_int2_row_quant_golden", "test_int2_row_quant_bounds"],
         [("const float s = amax / 1.0f;", "const float s = amax / 2.0f;")]),
    # the two record-offset mistakes read an int8 record at the int4 offsets, which stay inside
    # the record
    18: ("int8 expert records read at the int4 offsets", ["test_expert_of_equal_codes_is_the_same_in_every_width",
                                                          "test_int8_expert_against_fp64",
                                                          "test_layer_of_equal_codes_is_the_same_in_every_width"],
         [("const int64_t mat = (int64_t)f * d * bits / 8;",
           "const int64_t mat = (int64_t)f * d * (bits == 8 ? 4 : bits) / 8;")]),
    19: ("fp64 layer output reads down rows at the int4 offset", [
        "test_layer_of_equal_codes_is_the_same_in_every_width"],
         [("const int64_t down_at = 2 * ((int64_t)f * d * bits / 8);",
           "const int64_t down_at = 2 * ((int64_t)f * d * (bits == 8 ? 4 : bits) / 8);")]),
}


def mutant_source(n):
    """oracle.c with planted mistake n applied"""
    with open(os.path.join(O.HERE, "oracle.c")) as fh:
        src = fh.read()
    for trusted, planted in MUTANTS[n][2]:
        assert src.count(trusted) == 1, (n, trusted)
        src = src.replace(trusted, planted)
    return src


def write_mutant(n, directory):
    """the patched source of mutant n, written next to a copy of oracle.h in a directory of its
    own (so that mutants can be written and compiled in parallel); returns its path"""
    sub = os.path.join(str(directory), f"m{n}")
    os.makedirs(sub, exist_ok=True)
    path = os.path.join(sub, "oracle.c")
    with open(path, "w") as fh:
        fh.write(mutant_source(n))
    with open(os.path.join(O.HERE, "oracle.h")) as src, open(os.path.join(sub, "oracle.h"), "w") as dst:
        dst.write(src.read())
    return path


def test_every_patch_applies_once():
    for n in MUTANTS:
        assert mutant_source(n) != mutant_source(1 if n != 1 else 2)


@pytest.fixture
def mutant_lib(tmp_path):
    saved_so, saved_lib = O.SO, O._lib

    def use(n):
        so = str(tmp_path / f"liboracle_m{n}.so")
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off",
                               write_mutant(n, tmp_path), "-o", so, "-lm"])
        O.SO, O._lib = so, None
        O.lib()

    yield use
    O.SO, O._lib = saved_so, saved_lib


@pytest.mark.parametrize("n", sorted(MUTANTS))
def test_pin_catches_planted_mistake(n, mutant_lib):
    what, guards, _ = MUTANTS[n]
    mutant_lib(n)
    for name in guards:
        with pytest.raises(AssertionError):
            getattr(pins, name)()
