"""The pins catch plausible mistakes: each test plants one mistake in a COPY of the oracle's C
source (on the CPU), builds it, and checks that the pin aimed at that part of the method fails.
The oracle itself is never modified."""
import os
import subprocess

import numpy as np
import pytest

import oracle
import test_oracle as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "ep_oracle.c")

MUTATIONS = {
    # combine adds ranks in descending order instead of ascending
    "descending_rank_order": ("for (int r = 0; r < W; ++r) {                 /* ascending destination rank */",
                              "for (int r = W - 1; r >= 0; --r) {           /* planted */",
                              pins.test_combine_order_golden),
    # only the first top-k slot is routed
    "first_slot_only": ("                in_D[e / E] = 1;", "                if (j == 0) in_D[e / E] = 1;",
                        None),
    # reverse map drops the source rank
    "src_pos_without_rank": ("src_pos[(int64_t)r * rows + slot] = (int32_t)((int64_t)s * rows + t);",
                             "src_pos[(int64_t)r * rows + slot] = (int32_t)t;",
                             lambda: pins.test_dispatch_invariants(pins.CASES[0])),
    # BF16 conversion truncates instead of rounding to nearest even
    "bf16_truncation": ("    b += 0x7FFFu + kept_lsb;", "    b += 0u * kept_lsb;",
                        pins.test_bf16_rne_matches_torch_cast),
    # ties round away from zero instead of to even
    "bf16_ties_away": ("    b += 0x7FFFu + kept_lsb;", "    b += 0x8000u + 0u * kept_lsb;",
                       pins.test_bf16_rne_matches_torch_cast),
    # expert -> rank by modulo instead of contiguous blocks
    "rank_by_modulo": ("                in_D[e / E] = 1;", "                in_D[e % W] = 1;",
                       pins.test_brute_force_every_subset),
    # the weight rows are not summed (last one wins)
    "weights_overwrite": ("accw[j] = accw[j] + w_in[row * k + j];", "accw[j] = w_in[row * k + j];",
                          pins.test_combine_weights_dyadic_closed_form),
    # e4m3 saturation forgotten: values past 448 become NaN
    "e4m3_no_saturation": ("if (a >= 0x43E00000u) return (uint8_t)(sign | 0x7Eu);",
                           "if (a >= 0x43F00000u) return (uint8_t)(sign | 0x7Fu);",
                           pins.test_e4m3_rne_matches_torch_cast),
    # block scale uses the first element instead of the maximum
    "scale_not_amax": ("                if (m > amax) amax = m;", "                if (i == 0) amax = m;",
                       pins.test_blockwise_quantiser_properties),
    # FP8 wire dequantises with the wrong block's scale
    "wire_scale_index": ("* scales[row * nb + h / 128];", "* scales[row * nb];",
                         pins.test_fp8_combine_power_of_two_scales_closed_form),
    # e2m1 ties go to the odd code (away from even)
    "e2m1_ties_odd": ("if (dc < db || (dc == db && (c & 1) == 0)) best = c;",
                      "if (dc < db || (dc == db && (c & 1) == 1)) best = c;",
                      pins.test_e2m1_rne_brute_force),
    # e8m0 shared exponent off by one (largest e2m1 exponent taken as 1)
    "e8m0_off_by_one": ("                code = e2 - 2 + 127;", "                code = e2 - 1 + 127;",
                        pins.test_mxfp4_quantiser_against_numpy),
    # FP8 quotient formed as x times the rounded reciprocal of the scale, not the IEEE quotient
    "fp8_reciprocal_multiply": ("q[r * H + b * 128 + i] = ep_oracle_e4m3_from_f32(ep_oracle_f32_from_bf16(xb[i]) / scale);",
                                "q[r * H + b * 128 + i] = ep_oracle_e4m3_from_f32(ep_oracle_f32_from_bf16(xb[i]) * (1.0f / scale));",
                                pins.test_blockwise_quantiser_codes_are_the_ieee_quotient_cast),
    # e8m0 code 0 decoded as zero instead of the subnormal 2^-127
    "e8m0_code_zero_as_zero": ("if (c == 0) return bits_f32(0x00400000u);", "if (c == 0) return 0.0f;",
                               pins.test_e8m0_decode_every_code),
    # e8m0 code 0 decoded as 2^-126 (the exponent field read as if it were normal)
    "e8m0_code_zero_normal": ("if (c == 0) return bits_f32(0x00400000u);", "if (c == 0) return bits_f32(0x00800000u);",
                              pins.test_mxfp4_quantiser_tiny_blocks_take_scale_code_zero),
    # the FP4 combine pairs the wrong nibble with each element
    "fp4_nibble_swap": ("uint8_t code = (h & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xFu);",
                        "uint8_t code = (h & 1) ? (uint8_t)(byte & 0xFu) : (uint8_t)(byte >> 4);",
                        pins.test_fp4_combine_exact_sums),
    # grouped inverse sums in list order of the last expert only
    "ungroup_overwrite": ("acc[i * H + h] = acc[i * H + h] + v;", "acc[i * H + h] = v;",
                          pins.test_ungroup_identity_closed_form),
    # grouping: a source's first slot taken after its own rows (inclusive prefix)
    "layout_first_inclusive": ("                layout_range[list * W + s] = (first << 32) | per_src[s];\n"
                               "                first += per_src[s];",
                               "                first += per_src[s];\n"
                               "                layout_range[list * W + s] = (first << 32) | per_src[s];",
                               pins.test_group_by_expert_brute_force),
    # grouping: src_info keeps the source rank (the packed reverse-map entry, not the token)
    "src_info_with_rank": ("packed_src_info[list * rows + slot] = (int32_t)(pos % rows);",
                           "packed_src_info[list * rows + slot] = (int32_t)pos;",
                           pins.test_group_by_expert_brute_force),
    # grouping: only the last top-k entry is looked at
    "group_last_entry_only": ("for (int j = 0; j < k; ++j) named |= ids[j] == ge;",
                              "for (int j = 0; j < k; ++j) named = ids[j] == ge;",
                              pins.test_group_by_expert_brute_force),
}


@pytest.fixture(autouse=True)
def _restore():
    yield
    oracle.use_library(None)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new, pin = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = src.replace(old, new, 1)
    c = tmp_path / "mutant.c"
    c.write_text(mutated)
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                           "-o", str(so), str(c)])
    oracle.use_library(str(so))
    if pin is None:           # the exactly-once invariant over all cases
        pin = lambda: [pins.test_dispatch_invariants(c) for c in pins.CASES]  # noqa: E731
    with pytest.raises((AssertionError, ValueError)):
        pin()
