"""CPU tests of the fp64 oracle: every pin on the real oracle, and every
planted mistake in a copy of its source caught by at least one pin."""
import os

import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.default())


# (name, text in pa_oracle.c, replacement, count) -- count 0 replaces every occurrence.
MUTANTS = [
    ("gqa_modulo", "const int kh = h / (H / KH);", "const int kh = h % KH;", 0),
    ("slot_shifted", "int o = t % BS;", "int o = (t + 1) % BS;", 1),
    ("block_table_ignored", "bt[(size_t)s * MB + t / BS]", "bt[(size_t)s * MB + 0]", 1),
    ("key_read_as_value_layout",
     "return ((((size_t)b * KH + kh) * (D / x) + d / x) * BS + o) * x + d % x;",
     "(void)x; return (((size_t)b * KH + kh) * D + d) * BS + o;", 1),
    ("key_chunk_and_lane_swapped",
     "return ((((size_t)b * KH + kh) * (D / x) + d / x) * BS + o) * x + d % x;",
     "return ((((size_t)b * KH + kh) * (D / x) + d % (D / x)) * BS + o) * x + d / (D / x);", 1),
    ("value_transposed", "return (((size_t)b * KH + kh) * D + d) * BS + o;",
     "return (((size_t)b * KH + kh) * BS + o) * D + d;", 1),
    ("scale_dropped", "z[t - t0] = scale * acc;", "z[t - t0] = acc;", 1),
    ("exp_sign", "z[t] = exp(z[t] - mu);", "z[t] = exp(mu - z[t]);", 1),
    ("not_normalised", "for (int d = 0; d < D; ++d) o_sh[d] /= den;", "", 1),
    ("last_token_dropped", "int L = lens[s];\n        double* o_sh",
     "int L = lens[s] > 1 ? lens[s] - 1 : lens[s];\n        double* o_sh", 1),
    ("partition_end_short", "start + P < L ? start + P : L", "start + P - 1 < L ? start + P - 1 : L", 1),
    ("combine_without_l", "exp(m_sh[p] - M) * l_sh[p] / total", "exp(m_sh[p] - M) / total", 1),
    ("combine_total_without_l", "total += exp(m_sh[p] - M) * l_sh[p];", "total += exp(m_sh[p] - M);", 1),
    ("sentinel_max_zero", "m[shp] = -INFINITY; l[shp] = 0.0;", "m[shp] = 0.0; l[shp] = 0.0;", 1),
    ("fp16_exponent_bias", "expo - 25", "expo - 24", 1),
    ("bf16_shift", "((uint32_t)b) << 16", "((uint32_t)b) << 15", 1),
    ("lse_log2", "lse[sh] = mu + log(sum);", "lse[sh] = mu + log2(sum);", 1),
    ("lse_max_dropped", "lse[sh] = mu + log(sum);", "lse[sh] = log(sum);", 1),
    ("lse_exp_without_shift", "sum += exp(z[t] - mu);", "sum += exp(z[t]);", 1),
    ("combine_lse_without_l", "total += exp(m_sh[p] - M) * l_sh[p];\n        lse[sh]",
     "total += exp(m_sh[p] - M);\n        lse[sh]", 1),
    ("combine_lse_last_partition_dropped", "for (int p = 0; p < np; ++p) total += exp(m_sh[p] - M) * l_sh[p];\n        lse[sh]",
     "for (int p = 0; p + 1 < np; ++p) total += exp(m_sh[p] - M) * l_sh[p];\n        lse[sh]", 1),
    ("lse_empty_zero", "lse[sh] = -INFINITY;\n        if (L <= 0) continue;\n        if (L > MB * BS)",
     "lse[sh] = 0.0;\n        if (L <= 0) continue;\n        if (L > MB * BS)", 1),
    ("mq_not_causal", "const int visible = L - q_len + i + 1;", "const int visible = L;", 1),
    ("mq_causal_off_by_one", "const int visible = L - q_len + i + 1;", "const int visible = L - q_len + i;", 1),
    ("mq_rows_reversed", "const int visible = L - q_len + i + 1;", "const int visible = L - i;", 1),
    ("mq_first_query_row_only", "q + ((size_t)(s * q_len + i) * H + h) * D", "q + ((size_t)(s * q_len) * H + h) * D", 1),
    ("e4m3_bias", "ldexp((double)(8 + frac), expo - 10)", "ldexp((double)(8 + frac), expo - 11)", 1),
    ("e4m3_subnormal_scale", "v = ldexp((double)frac, -9);", "v = ldexp((double)frac, -10);", 1),
    ("e4m3_no_nan_rule", "if (expo == 15 && frac == 7) {", "if (0) {", 1),
    ("fp8_k_scale_dropped", "(k_scale * e4m3_to_double(", "(1.0 * e4m3_to_double(", 1),
    ("fp8_v_scale_dropped", "(v_scale * e4m3_to_double(", "(1.0 * e4m3_to_double(", 1),
    ("fp8_key_x8", "    const int x = 16;\n    return", "    const int x = 8;\n    return", 1),
    ("mq_fp8_not_causal", "const int seen = L - q_len + i + 1;", "const int seen = L;", 1),
    ("mq_fp8_causal_off_by_one", "const int seen = L - q_len + i + 1;", "const int seen = L - q_len + i;", 1),
    ("mq_fp8_first_query_row_only", "const uint16_t* qrow = q + ((size_t)(s * q_len + i) * H + h) * D;",
     "const uint16_t* qrow = q + ((size_t)(s * q_len) * H + h) * D;", 1),
    ("mq_fp8_k_scale_dropped", "acc += to_double(qrow[d], qdtype) *\n                       (k_scale *",
     "acc += to_double(qrow[d], qdtype) *\n                       (1.0 *", 1),
    ("mq_fp8_v_scale_dropped", "o_r[d] += z[t] * (v_scale *", "o_r[d] += z[t] * (1.0 *", 1),
    ("mq_fp8_value_read_with_key_layout", "o_r[d] += z[t] * (v_scale * e4m3_to_double(vc[value_index(",
     "o_r[d] += z[t] * (v_scale * e4m3_to_double(vc[key_index_x16(", 1),
    ("fp32_key_x8", "    const int x = 4;\n    return", "    const int x = 8;\n    return", 1),
    ("fp32_key_read_as_value", "(double)kc[key_index_x4(b, kh, d, o, KH, D, BS)]",
     "(double)kc[value_index(b, kh, d, o, KH, D, BS)]", 1),
    ("fp32_weights_dropped", "o_sh[d] += z[t] * (double)vc[", "o_sh[d] += (double)vc[", 1),
    ("mq_fp32_not_causal", "const int upto = L - q_len + i + 1;", "const int upto = L;", 1),
    ("mq_fp32_causal_off_by_one", "const int upto = L - q_len + i + 1;", "const int upto = L - q_len + i;", 1),
    ("mq_fp32_first_query_row_only", "const float* qr = q + ((size_t)(s * q_len + i) * H + h) * D;",
     "const float* qr = q + ((size_t)(s * q_len) * H + h) * D;", 1),
    ("mq_fp32_key_read_as_value", "(double)qr[d] * (double)kc[key_index_x4(",
     "(double)qr[d] * (double)kc[value_index(", 1),
    ("mq_fp32_weights_dropped", "o_r[d] += z[t] * (double)vc[", "o_r[d] += (double)vc[", 1),
    ("empty_sequence_not_zero", "if (L <= 0) continue;\n        if (L > MB * BS) { bad = 1; continue; }\n        double* z",
     "if (L > MB * BS) { bad = 1; continue; }\n        double* z", 1),
]


def _run_pins(orc):
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError, FloatingPointError) as e:
            failed.append((pin.__name__, str(e)[:80]))
    return failed


@pytest.mark.parametrize("name,old,new,count", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new, count):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "pa_oracle.c")).read()
    assert old in src, f"mutation target for {name} not found in the oracle source"
    mutated = src.replace(old, new) if count == 0 else src.replace(old, new, count)
    path = tmp_path / "mutant.c"
    path.write_text(mutated)
    so = oracle.build(force=True, src=str(path), out=str(tmp_path / "libmutant.so"))
    failed = _run_pins(oracle.Oracle(oracle.load_library(so)))
    assert failed, f"planted mistake '{name}' passed every pin"
