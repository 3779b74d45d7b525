"""Plant plausible mistakes in copies of the oracle (on the CPU) and check
that the pins catch every one of them: a dropped term, a wrong index or
sign, a reversed loop, a wrong start value, a different rounding.

Each mutant is one textual replacement in a temporary copy of
``oracle/mp_oracle.c``; the copy is compiled with the oracle's own flags and
loaded next to the real one.  Mutants are chosen so that none of them
writes outside its buffers.
"""
import os

import pytest

import oracle
from tests import pins

MUTANTS = {
    "round_half_up": ("if (dropped > half ||", "if (dropped >= half ||"),
    "ties_to_odd": ("(dropped == half && (kept & 1u))", "(dropped == half && !(kept & 1u))"),
    "widen_wrong_shift": ("((uint32_t)b) << 16", "((uint32_t)b) << 15"),
    "owner_round_robin": ("mask |= 1u << (e / El);", "mask |= 1u << (e % R);"),
    "expert_count_mirrored": ("num_tokens_per_expert[(int64_t)s * E + e] += 1;",
                              "num_tokens_per_expert[(int64_t)s * E + (E - 1 - e)] += 1;"),
    "masked_counts_as_rank0": ("if (e == -1) continue; /* masked entry */",
                               "if (e == -1) { mask |= 1u; continue; }"),
    "tokens_descending": ("for (int t = 0; t < N; ++t) {\n        const int64_t tok = (int64_t)s * N + t;\n        if (!((is_token_in_rank",
                          "for (int t = N - 1; t >= 0; --t) {\n        const int64_t tok = (int64_t)s * N + t;\n        if (!((is_token_in_rank"),
    "global_expert_ids": ("local ? e - d * El : -1", "local ? e : -1"),
    "nonlocal_weight_kept": ("local ? topk_weights[tok * K + k] : 0.0f", "topk_weights[tok * K + k]"),
    "rank_prefix_absolute": ("rank_prefix[(int64_t)s * R + d] = (int32_t)(row - dest_offsets[d]);",
                             "rank_prefix[(int64_t)s * R + d] = (int32_t)(row);"),
    "src_idx_off_by_one": ("recv_src_idx[row] = t;", "recv_src_idx[row] = t + 1;"),
    "recv_expert_count_shifted": ("if (e >= 0 && e < E) num_recv_tokens_per_expert[e] += 1;",
                                  "if (e >= 0 && e < E) num_recv_tokens_per_expert[(e + 1) % E] += 1;"),
    "combine_descending": ("for (int d = 0; d < R; ++d) {\n        int32_t r = send_row",
                           "for (int d = R - 1; d >= 0; --d) {\n        int32_t r = send_row"),
    "combine_negative_zero_start": ("const int64_t tok = (int64_t)s * N + t;\n      for (int h = 0; h < H; ++h) acc[h] = 0.0f;",
                                    "const int64_t tok = (int64_t)s * N + t;\n      for (int h = 0; h < H; ++h) acc[h] = -0.0f;"),
    "combine_drops_first_rank": ("if (r < 0) continue;\n        if ((int64_t)r >= y_rows)",
                                 "if (r < 0 || d == 0) continue;\n        if ((int64_t)r >= y_rows)"),
    "combine_in_double": ("R > 32 || N < 0 || H < 0 || y_rows < 0) return ORC_BAD_ARG;\n  int status = 0;\n  float *acc = (float *)malloc(sizeof(float)",
                          "R > 32 || N < 0 || H < 0 || y_rows < 0) return ORC_BAD_ARG;\n  int status = 0;\n  double *acc = (double *)malloc(sizeof(double)"),
    "rsv_descending": ("for (int q = 0; q < R; ++q)\n          acc = acc",
                       "for (int q = R - 1; q >= 0; --q)\n          acc = acc"),
    "rsv_in_double": ("        float acc = 0.0f;\n        for (int q = 0; q < R; ++q)",
                      "        double acc = 0.0;\n        for (int q = 0; q < R; ++q)"),
    "e4m3_ties_away": ("if (rem > half || (rem == half && (q & 1u))) q += 1u;",
                       "if (rem >= half) q += 1u;"),
    "e4m3_bias_off": ("(uint8_t)((e + 7) << 3)", "(uint8_t)((e + 8) << 3)"),
    "e4m3_no_subnormals": ("uint32_t k = rne_shift(sig, 23 - (e + 9)); /* in [0, 8] */",
                           "uint32_t k = 0u; (void)rne_shift; /* flushed */"),
    "quant_divisor_240": ("amax > 0.0f ? amax / 448.0f : 1.0f", "amax > 0.0f ? amax / 240.0f : 1.0f"),
    "quant_multiplies": ("oracle_f32_to_e4m3(oracle_bf16_to_f32(xb[h]) / scale)",
                         "oracle_f32_to_e4m3(oracle_bf16_to_f32(xb[h]) * scale)"),
    "quant_reciprocal_first": ("oracle_f32_to_e4m3(oracle_bf16_to_f32(xb[h]) / scale)",
                               "oracle_f32_to_e4m3(oracle_bf16_to_f32(xb[h]) * (1.0f / scale))"),
    "quant_zero_scale": ("amax > 0.0f ? amax / 448.0f : 1.0f", "amax > 0.0f ? amax / 448.0f : 0.0f"),
    "global_ids_sentinel_ignored": ("(e >= d * El && e < (d + 1) * El) ? e : sentinel;",
                                    "(e >= d * El && e < (d + 1) * El) ? e : -1;"),
    "global_ids_off_by_rank": ("for (int d = 0; d < R; ++d) {\n    for (int64_t r = dest_offsets[d]; r < dest_offsets[d + 1]; ++r) {",
                               "for (int d = 0; d < R; ++d) {\n    for (int64_t r = dest_offsets[d]; r < dest_offsets[d + 1] - (d == 0); ++r) {"),
    "combined_weights_skip_last": ("        acc = acc + recv_topk_weights[(int64_t)r * K + k];",
                                   "        if (d < R - 1) acc = acc + recv_topk_weights[(int64_t)r * K + k];"),
    "ll_source_major": ("  for (int e = 0; e < E; ++e) {\n    expert_offsets[e] = (int32_t)row;\n    for (int s = 0; s < R; ++s) {",
                        "  for (int e = E - 1; e >= 0; --e) {\n    expert_offsets[e] = (int32_t)row;\n    for (int s = 0; s < R; ++s) {"),
    "ll_unweighted": ("const float p = w * oracle_bf16_to_f32(y[(int64_t)r * H + h]);",
                      "const float p = oracle_bf16_to_f32(y[(int64_t)r * H + h]);"),
    "ll_keeps_masked": ("if (topk_idx[tok * K + k] != e) continue;",
                        "if (topk_idx[tok * K + k] != e && !(e == 0 && topk_idx[tok * K + k] == -1)) continue;"),
    "mxfp8_emax_7": ("code = floor_log2_f32(amax) - 8 + 127;", "code = floor_log2_f32(amax) - 7 + 127;"),
    "mxfp8_flush_tiny": ("- 8 + 127;\n        if (code < 0) code = 0;\n", "- 8 + 127;\n        if (code < 0) code = 0, amax = 0.0f;\n        if (amax == 0.0f) { for (int h = 0; h < 32; ++h) q[t * H + (int64_t)b * 32 + h] = 0; codes[t * nb + b] = 0; continue; }\n"),
    "e2m1_ties_up": ("if (dc < db || (dc == db && (c & 1) == 0)) best = c;",
                     "if (dc <= db) best = c;"),
    "e2m1_sign_dropped": ("const uint8_t sign = signbit(x) ? 8u : 0u;",
                          "const uint8_t sign = 0u;"),
    "mxfp4_emax_8": ("code = floor_log2_f32(amax) - 2 + 127;", "code = floor_log2_f32(amax) - 8 + 127;"),
    "mxfp4_nibbles_swapped": ("qb[h / 2] = (uint8_t)(lo | (hi << 4));", "qb[h / 2] = (uint8_t)(hi | (lo << 4));"),
    "e2m1_saturates_to_4": ("if (!(a < 6.0)) return (uint8_t)(sign | 7u);", "if (!(a < 6.0)) return (uint8_t)(sign | 6u);"),
    "ll_rank_major_by_expert_owner_mod": ("if (e < d * El || e >= (d + 1) * El) continue;",
                                          "if (e % R != d) continue;"),
    "ll_rank_major_slot_order_dropped": ("for (int t = 0; t < N; ++t) {\n        const int64_t tok = (int64_t)s * N + t;\n        for (int k = 0; k < K; ++k) {\n          const int e = topk_idx[tok * K + k];",
                                         "for (int t = N - 1; t >= 0; --t) {\n        const int64_t tok = (int64_t)s * N + t;\n        for (int k = 0; k < K; ++k) {\n          const int e = topk_idx[tok * K + k];"),
    "ll_rank_major_src_offsets_absolute": ("dest_src_offsets[d * R + s] = (int32_t)(row - dest_offsets[d]);",
                                           "dest_src_offsets[d * R + s] = (int32_t)(row);"),
    "agv_shard_shift": ("memcpy(out + ((int64_t)q * S + i) * row_bytes, in + i * row_bytes",
                        "memcpy(out + ((int64_t)q * S + i) * row_bytes, in + (i - off) * row_bytes"),
    "ll_combine_descending": ("    for (int k = 0; k < K; ++k) {\n      const int32_t r = slot_row[tok * K + k];",
                              "    for (int k = K - 1; k >= 0; --k) {\n      const int32_t r = slot_row[tok * K + k];"),
    "ll_combine_fused_multiply_add": ("        acc[h] = acc[h] + p;",
                                      "        acc[h] = fmaf(w, oracle_bf16_to_f32(y[(int64_t)r * H + h]), acc[h]);"),
    "capacity_row_not_advanced": ("if (row >= recv_capacity) { status |= ORC_CAPACITY; row += 1; continue; }",
                                  "if (row >= recv_capacity) { status |= ORC_CAPACITY; continue; }"),
    "scales_from_first_token": ("          recv_scales[row * scales_per_row + c] = x_scales[tok * scales_per_row + c];",
                                "          recv_scales[row * scales_per_row + c] = x_scales[c];"),
    "combine_capacity_not_flagged": ("        if ((int64_t)r >= y_rows) { status |= ORC_CAPACITY; continue; }\n        const uint16_t *src = y",
                                     "        if ((int64_t)r >= y_rows) { continue; }\n        const uint16_t *src = y"),
    "combined_weights_capacity_not_flagged": ("        if ((int64_t)r >= recv_rows) { status |= ORC_CAPACITY; continue; }\n        acc = acc + recv_topk_weights",
                                              "        if ((int64_t)r >= recv_rows) { continue; }\n        acc = acc + recv_topk_weights"),
    "combined_weights_descending": ("      for (int d = 0; d < R; ++d) {\n        const int32_t r = send_row[tok * R + d];\n        if (r < 0) continue;\n        if ((int64_t)r >= recv_rows)",
                                    "      for (int d = R - 1; d >= 0; --d) {\n        const int32_t r = send_row[tok * R + d];\n        if (r < 0) continue;\n        if ((int64_t)r >= recv_rows)"),
    "ll_capacity_not_flagged": ("          } else {\n            status |= ORC_CAPACITY;\n          }\n          row += 1;\n        }\n      }\n    }\n  }\n  expert_offsets[E]",
                                "          } else {\n          }\n          row += 1;\n        }\n      }\n    }\n  }\n  expert_offsets[E]"),
    "ll_capacity_row_not_advanced": ("          } else {\n            status |= ORC_CAPACITY;\n          }\n          row += 1;\n        }\n      }\n    }\n  }\n  expert_offsets[E]",
                                     "          } else {\n            status |= ORC_CAPACITY; row -= 1;\n          }\n          row += 1;\n        }\n      }\n    }\n  }\n  expert_offsets[E]"),
    "rsv_negative_zero_start": ("        float acc = 0.0f;\n        for (int q = 0; q < R; ++q)",
                                "        float acc = -0.0f;\n        for (int q = 0; q < R; ++q)"),
    "bf16_nan_quiet_bit_dropped": ("return (uint16_t)((u >> 16) | 0x0040u);",
                                   "return (uint16_t)(u >> 16);"),
}


@pytest.fixture(scope="module")
def src_text():
    with open(os.path.join(os.path.dirname(oracle.__file__), "mp_oracle.c")) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, src_text, tmp_path):
    old, new = MUTANTS[name]
    assert src_text.count(old) == 1, "mutation site not unique: %s" % name
    src = tmp_path / ("mut_%s.c" % name)
    src.write_text(src_text.replace(old, new))
    lib = oracle.compile_oracle(str(src), str(tmp_path / ("libmut_%s.so" % name)))
    orc = oracle.OracleLib(lib)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            caught.append(pin.__name__)
            break
    assert caught, "no pin caught the planted mistake %r" % name
