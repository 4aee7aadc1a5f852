"""Plant one plausible mistake at a time in a copy of the oracle's C source,
build it, and check that at least one pin fails.  This is what makes the pins
worth trusting: a dropped term, a wrong sign or index, a transposed operand
or a wrong rounding rule anywhere in the oracle does not go unnoticed.
CPU only; the real oracle is never modified."""
import pytest

import oracle
import oracle_pins as pins

# (name, text in moe_oracle.c, replacement)
MUTANTS = [
    ("gate_up_swapped", "a[j] = silu(g) * u;", "a[j] = silu(u) * g;"),
    ("silu_dropped", "a[j] = silu(g) * u;", "a[j] = g * u;"),
    ("silu_sign", "return g / (1.0 + exp(-g));", "return g / (1.0 + exp(g));"),
    ("sigmoid_not_silu", "return g / (1.0 + exp(-g));", "return 1.0 / (1.0 + exp(-g));"),
    ("routing_weight_dropped", "o[c] += w * y[c];", "o[c] += y[c];"),
    ("slot_index_k_dropped", "int e = ids[(size_t)t * p->K + k];",
     "int e = ids[(size_t)t * p->K];"),
    ("weight_index_wrong", "double w = (double)topk_w[(size_t)t * p->K + k];",
     "double w = (double)topk_w[(size_t)k];"),
    ("down_proj_wrong_expert", "expert_out(p, w2, w2_scale, e, a, y, wrow);\n            for (int c = 0; c < p->H; ++c) o[c]",
     "expert_out(p, w2, w2_scale, 0, a, y, wrow);\n            for (int c = 0; c < p->H; ++c) o[c]"),
    ("up_row_offset_wrong", "2 * j + 1 : p->I + j;", "2 * j + 1 : (j + 1 < p->I ? j + 1 : j);"),
    ("bf16_decode_shift", "((uint32_t)b) << 16", "((uint32_t)b) << 15"),
    ("e2m1_exponent_bias", "ldexp(1.0 + 0.5 * m, e - 1)", "ldexp(1.0 + 0.5 * m, e)"),
    ("e8m0_bias", "ldexp(1.0, (int)v - 127)", "ldexp(1.0, (int)v - 128)"),
    ("e4m3_bias", "ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    ("mx_nibble_order", "(c & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15)",
     "(c & 1) ? (uint8_t)(byte & 15) : (uint8_t)(byte >> 4)"),
    ("mx_scale_block_64", "sc[c / 32]", "sc[c / 64]"),
    ("e4m3_ties_toward_zero", "(err == best_err && (c & 1) == 0 && (best & 1) == 1)", "0"),
    ("x_scale_divisor", "amax / 448.0f", "amax / 256.0f"),
    ("align_unstable_order",
     "for (long i = 0; i < na; ++i) {\n            if (ids[i] != e) continue;",
     "for (long i = na - 1; i >= 0; --i) {\n            if (ids[i] != e) continue;"),
    # under-padding keeps every write inside the buffers (over-padding would not)
    ("align_padding_rule", "(counts[e] + bm - 1) / bm * bm", "counts[e] / bm * bm"),
    ("align_sentinel", "sorted_ids[s] = (int32_t)na;", "sorted_ids[s] = -1;"),
    ("align_valid_rows", "bi[3] = left < bm ? left : bm;", "bi[3] = bm;"),
    ("align_bad_id_accepted", "if (ids[i] < 0 || ids[i] >= E) return -1;\n    for (int e = 0; e < L; ++e) counts[e] = 0;",
     "for (int e = 0; e < L; ++e) counts[e] = 0;"),
    ("combine_slot_index", "int slot = inv_perm[(size_t)t * K + k];",
     "int slot = inv_perm[(size_t)t * K];"),
    ("gather_row_index", "load_token_row(p, x, i / p->K, xrow);",
     "load_token_row(p, x, i % p->T, xrow);"),
    ("swiglu_alpha_dropped", "exp(-p->swiglu_alpha * g)", "exp(-g)"),
    ("swiglu_plus_one_dropped", "* (u + 1.0);", "* u;"),
    ("swiglu_gate_clamped_below", "g = fmin(g, p->swiglu_limit);",
     "g = fmax(fmin(g, p->swiglu_limit), -p->swiglu_limit);"),
    ("swiglu_linear_not_clamped_below", "u = fmax(fmin(u, p->swiglu_limit), -p->swiglu_limit);",
     "u = fmin(u, p->swiglu_limit);"),
    ("swiglu_up_takes_gate_bias", "(b13 ? (double)b13[up_row(p, j)] : 0.0)",
     "(b13 ? (double)b13[gate_row(p, j)] : 0.0)"),
    ("interleaved_gate_row_wrong", "return p->gate_up_interleaved ? 2 * j : j;",
     "return p->gate_up_interleaved ? 2 * j + 1 : j;"),
    ("w2_bias_dropped", " + (p->w2_bias ? (double)p->w2_bias[(size_t)e * p->H + c] : 0.0)", ""),
    ("route_ties_to_higher_id", "if (best < 0 || l > bv) {", "if (best < 0 || l >= bv) {"),
    ("route_softmax_over_first_only", "for (int k = 0; k < K; ++k) sum += exp(v[k] - v[0]);",
     "for (int k = 0; k < K; ++k) sum += exp(v[0] - v[0]);"),
    ("route_keeps_taken", "if (taken[e]) continue;", "if (0) continue;"),
    ("shard_other_slots_keep_slot", "        inv_perm[i] = -1;\n", "        inv_perm[i] = 0;\n"),
    ("h_scale_multiplies_in_store", "float q = (float)(a / p->h_scale);",
     "float q = (float)(a * p->h_scale);"),
    ("h_scale_dropped_in_store", "return orc_e4m3_to_double(orc_float_to_e4m3(q)) * p->h_scale;",
     "return orc_e4m3_to_double(orc_float_to_e4m3(q));"),
    ("h_scale_twice_in_store", "return orc_e4m3_to_double(orc_float_to_e4m3(q)) * p->h_scale;",
     "return orc_e4m3_to_double(orc_float_to_e4m3(q)) * p->h_scale * p->h_scale;"),
    ("h_scale_dropped_in_down",
     "a[j] = orc_e4m3_to_double(((const uint8_t*)hin)[base + j]) * p->h_scale;",
     "a[j] = orc_e4m3_to_double(((const uint8_t*)hin)[base + j]);"),
    ("bf16_rounds_through_fp32", "double r = ldexp(rint(ldexp(v, -q)), q);",
     "double r = ldexp(rint(ldexp((double)(float)v, -q)), q);"),
    ("bf16_ties_away_from_zero", "double r = ldexp(rint(ldexp(v, -q)), q);",
     "double r = ldexp(round(ldexp(v, -q)), q);"),
    ("shard_weight_index_global", "e -= p->expert_base; /* index into this shard's weights */",
     "e = e % shard_size(p);"),
]

ALL_PINS = pins.FORMAT_PINS + [pins.pin_align_rejects_bad_id, pins.pin_align_invariants] + [
    (lambda c=c: pins.pin_align_vs_stable_argsort(*c)) for c in pins.ALIGN_CASES[:7]
] + pins.FFN_PINS + pins.SHARD_PINS + pins.SWIGLU_PINS + pins.ROUTE_PINS


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(mutant, tmp_path):
    name, old, new = mutant
    src = oracle.source()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    so = oracle.build_variant(src.replace(old, new, 1), str(tmp_path), name)
    with oracle.using_library(so):
        for pin in ALL_PINS:
            try:
                pin()
            except Exception:  # an assertion, or a pin's own indexing tripping on bad output
                return  # caught
    pytest.fail(f"no pin caught the planted mistake {name}")
