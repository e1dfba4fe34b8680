"""Plant plausible mistakes in copies of the oracle and check a pin catches each.

Every mutant is a textual edit of the oracle's C source, compiled into a
temporary library (CPU only).  A mutant that no pin rejects would mean the
pins leave that part of the oracle unchecked.
"""
import os

import pytest

import oracle as oracle_mod
import pins

MUTANTS = {
    "dropped_scale": [("scores[t] = scale * dot;", "scores[t] = dot;")],
    "in_block_offset": [("return block * bs + t % bs;", "return block * bs + (t + 1) % bs;")],
    "block_index": [("block_tables[(int64_t)b * max_nb + t / bs]",
                     "block_tables[(int64_t)b * max_nb + (t / bs + 1) % max_nb]")],
    "gqa_interleaved": [("int32_t n = kvh * G + g;", "int32_t n = g * j->K + kvh;")],
    "no_max_subtraction": [("scores[t] = exp(scores[t] - mx);", "scores[t] = exp(scores[t]);"),
                           ("*lse = mx + log(sum);", "*lse = log(sum);")],
    "keys_for_values": [("acc += scores[t] * values[t * H + h];",
                         "acc += scores[t] * keys[t * H + h];")],
    "context_off_by_one": [("const int64_t ctx = j->context_lens[b] > 0 ? j->context_lens[b] : 0;",
                            "const int64_t ctx = j->context_lens[b] > 1 ? j->context_lens[b] - 1 : 0;")],
    "lse_missing_log": [("*lse = mx + log(sum);", "*lse = mx + sum;")],
    "merge_weight_sign": [("acc += exp(pl[p] - total) * part_out",
                           "acc += exp(total - pl[p]) * part_out")],
    "append_token_order": [("memcpy(k_cache + (size_t)slots[i] * row, k_new + (size_t)i * row,",
                            "memcpy(k_cache + (size_t)slots[i] * row, k_new + (size_t)(T - 1 - i) * row,")],
    "slot_mapping_off_by_one": [("int64_t pos = (int64_t)context_lens[b] - 1;",
                                 "int64_t pos = (int64_t)context_lens[b] - 2;")],
    "bf16_widening": [("uint32_t bits = (uint32_t)bits16 << 16;",
                       "uint32_t bits = ((uint32_t)bits16 << 16) | 0x8000u;")],
    "gather_neighbour": [("int64_t slot = physical_slot(block_tables, max_nb, b, t, bs);",
                          "int64_t slot = physical_slot(block_tables, max_nb, b, t ^ 1, bs);")],
    "partition_drops_token": [("int64_t t1 = t0 + j->partition_tokens;",
                               "int64_t t1 = t0 + j->partition_tokens - 1;")],
    "kv_bytes_factor": [("return 2u * (uint64_t)layers", "return 1u * (uint64_t)layers")],
    "e4m3_bias": [("ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)")],
    "e4m3_round_half_up": [("double r = nearbyint(a / quantum);", "double r = floor(a / quantum + 0.5);")],
    "e4m3_no_saturation": [("if (a >= 448.0) return (uint8_t)(sign | 0x7E);", "if (a >= 480.0) return (uint8_t)(sign | 0x7E);")],
    "e4m3_subnormal_quantum": [("const double quantum = ldexp(1.0, e - 3);", "const double quantum = ldexp(1.0, e - 3 + (e == -6));")],
    "fp8_scale_multiplies": [("dst[i] = oracle_e4m3_encode(x / sc[kvh]);", "dst[i] = oracle_e4m3_encode(x * sc[kvh]);")],
    "fp8_v_scale_for_k": [("keys[t * H + h] = oracle_e4m3_decode(j->k8[row + h]) * (double)j->k_scale[si];",
                           "keys[t * H + h] = oracle_e4m3_decode(j->k8[row + h]) * (double)j->v_scale[si];")],
    "fp8_block_scale_of_logical_block": [("(size_t)(slot / j->bs) * (size_t)j->scale_block_stride",
                                          "(size_t)(t / j->bs) * (size_t)j->scale_block_stride")],
    "fp8_quantize_ignores_block": [("scale + (scale_block_stride ? (size_t)(r / bs) * (size_t)scale_block_stride : 0)",
                                    "scale")],
    "fp8_append_scale_of_wrong_block": [("(size_t)(slots[i] / bs) * (size_t)scale_block_stride",
                                         "(size_t)(slots[i] % bs) * (size_t)scale_block_stride")],
    "multi_mask_top_left": [("int64_t visible = ctx - T + t + 1;", "int64_t visible = t + 1;")],
    "multi_mask_off_by_one": [("int64_t visible = ctx - T + t + 1;", "int64_t visible = ctx - T + t;")],
    "multi_query_row": [("const uint16_t *qrow = j->q + bn * H;",
                         "const uint16_t *qrow = j->q + ((size_t)b * T * j->N + n) * H;")],
    "slot_multi_offset": [("int64_t pos = (int64_t)context_lens[b] - T + t;",
                           "int64_t pos = (int64_t)context_lens[b] - T + t + 1;")],
    "copy_blocks_reversed": [("const int64_t src = src_dst[2 * i], dst = src_dst[2 * i + 1];",
                              "const int64_t dst = src_dst[2 * i], src = src_dst[2 * i + 1];")],
    "copy_blocks_k_only": [("v_cache[dst * block_bytes + x] = v_cache[src * block_bytes + x];", "")],
    "weights_not_normalised": [("for (int64_t t = 0; t < ntok; ++t) scores[t] /= sum;",
                                "for (int64_t t = 0; t < ntok; ++t) scores[t] /= (double)ntok;")],
}


def _caught(orc):
    failed = []
    for check in pins.ALL_CHECKS:
        try:
            check(orc)
        except (AssertionError, ValueError, FloatingPointError):
            failed.append(check.__name__)
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(tmp_path, name):
    src = open(oracle_mod.SOURCE, encoding="utf-8").read()
    for old, new in MUTANTS[name]:
        assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
        src = src.replace(old, new)
    path = tmp_path / "mutant.c"
    path.write_text(src, encoding="utf-8")
    lib = oracle_mod.compile_oracle(str(path), str(tmp_path / f"lib_{name}.so"))
    failed = _caught(oracle_mod.Oracle(lib))
    assert failed, f"no pin rejects the mutant {name}"
