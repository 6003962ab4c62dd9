"""Planted mistakes: each test compiles a copy of the C oracle with one
plausible mistake (a wrong index, a dropped term, a swapped operand, another
rounding) and checks that the pins reject it.  The mistakes are planted in
the oracle, on the CPU, in a temporary copy; the real oracle is untouched."""
import ctypes
import subprocess

import pytest

import oracle
from test_oracle_append import check_fp32_decision, check_rounding
from test_oracle_attention import (check_against_sdpa, check_int8_against_sdpa, check_online,
                                   check_partials_merge, small)
from test_oracle_fp8 import check_decode, check_encode, check_fp8_against_sdpa, check_saturation
from test_oracle_multi import check_multi_against_sdpa, multi


def _sdpa():
    check_against_sdpa(small([1, 2, 3, 15, 16, 17, 31, 33, 100, 250], hq=8, hkv=2, d=64, bs=16, seed=11))


def _sdpa_int8():
    check_int8_against_sdpa(small([1, 5, 32, 33, 70, 200], hq=16, hkv=2, d=128, bs=32, kv="int8", seed=3))


def _sdpa_fp8():
    check_fp8_against_sdpa(small([1, 5, 32, 33, 70, 200], hq=16, hkv=2, d=128, bs=32, kv="fp8", seed=3))


def _fp8_codes():
    check_decode(oracle.fp8_value)
    check_encode(oracle.quantize_fp8)
    check_saturation(oracle.quantize_fp8)


def _multi():
    check_multi_against_sdpa(multi([1, 5, 17, 40, 100, 250], [1, 5, 3, 40, 7, 64], hq=8, hkv=2, d=64))


def _online():
    check_online(16)


def _merge():
    for part in (16, 48, 512):
        check_partials_merge(part)


def _rounding():
    check_rounding(oracle.quantize_int8)


def _fp32():
    check_fp32_decision(oracle.quantize_int8)


MUTANTS = {
    "gqa_modulo_mapping": ("int hk = h / (P->num_q_heads / P->num_kv_heads);",
                           "int hk = h % P->num_kv_heads;", _sdpa),
    "row_off_by_one": ("K[(int64_t)t * d + e] = pool_value(P, 0, block, t % bs, hk, e);",
                       "K[(int64_t)t * d + e] = pool_value(P, 0, block, (t + 1) % bs, hk, e);", _sdpa),
    "scale_dropped": ("s[t] = P->scale * acc;", "s[t] = acc;", _sdpa),
    "v_reads_k": ("V[(int64_t)t * d + e] = pool_value(P, 1, block",
                  "V[(int64_t)t * d + e] = pool_value(P, 0, block", _sdpa),
    "last_token_dropped": ("for (int t = 0; t < L; ++t) {\n        double w = exp(s[t] - m) / Z;",
                           "for (int t = 0; t < L - 1; ++t) {\n        double w = exp(s[t] - m) / Z;", _sdpa),
    "table_index_transposed": ("P->block_tables[(int64_t)b * P->max_blocks + t / bs]",
                               "P->block_tables[(int64_t)b * P->max_blocks + t % bs]", _sdpa),
    "slot_row_wrong": ("slots[i] = (int64_t)physical * block_size + (p % block_size);",
                       "slots[i] = (int64_t)physical * block_size + (p / block_size);", _sdpa),
    "sum_sign_flipped": ("Z += exp(s[t] - m);", "Z += exp(m - s[t]);", _sdpa),
    "dequant_scale_dropped": ("return (double)c[idx] * sc;", "return (double)c[idx];", _sdpa_int8),
    "fp8_dequant_scale_dropped": ("return oracle_fp8_value(c[idx]) * sc;",
                                  "return oracle_fp8_value(c[idx]);", _sdpa_fp8),
    "fp8_ties_to_odd": ("(d == best_d && (c & 1) == 0)", "(d == best_d && (c & 1) == 1)", _fp8_codes),
    "fp8_exponent_bias_8": ("ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)", _fp8_codes),
    "fp8_subnormal_exponent": ("ldexp(m / 8.0, -6)", "ldexp(m / 8.0, -7)", _fp8_codes),
    "fp8_no_saturation": ("        return sign | 0x7E;", "        return 0x7F;", _fp8_codes),
    "fp8_sign_dropped": ("    return sign | (uint8_t)best;", "    return (uint8_t)best;", _fp8_codes),
    "multi_excludes_own_token": ("*L_out = L - n + (j - qs[b]) + 1;", "*L_out = L - n + (j - qs[b]);",
                                 _multi),
    "multi_sees_one_more": ("*L_out = L - n + (j - qs[b]) + 1;",
                            "*L_out = L - n + (j - qs[b]) + 1 + (j - qs[b] + 1 < n);", _multi),
    "multi_query_row_of_sequence": ("qrow = (int64_t)j * P->num_q_heads + h;",
                                    "qrow = (int64_t)b * P->num_q_heads + h;", _multi),
    "online_carry_dropped": ("double l_new = l_old * carry + sum;", "double l_new = l_old + sum;",
                             _online),
    "online_output_not_rescaled": ("o[e] = o[e] * l_old * carry / l_new + num[e] / l_new;",
                                   "o[e] = o[e] + num[e] / l_new;", _online),
    "partition_end_off_by_one": ("t1 = (i + 1) * part < L ? (i + 1) * part : L;",
                                 "t1 = (i + 1) * part < L ? (i + 1) * part - 1 : L;", _merge),
    "partial_sum_of_scores": ("            l += p;\n", "            l += s[t];\n", _merge),
    "merge_denominator_unweighted": ("den += w * ml[2 * i + 1];", "den += ml[2 * i + 1];", _merge),
    "merge_weight_sign_flipped": ("double w = exp(ml[2 * i] - M);", "double w = exp(M - ml[2 * i]);",
                                  _merge),
    "round_half_away": ("float r = nearbyintf(x / s);", "float r = roundf(x / s);", _rounding),
    "fp64_decision": ("float r = nearbyintf(x / s);",
                      "float r = (float)nearbyint((double)x / (double)s);", _fp32),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(oracle_mod, tmp_path, name):
    old, new, check = MUTANTS[name]
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, "mutation site not found"
    c = tmp_path / "mutant.c"
    c.write_text(src.replace(old, new))
    so = tmp_path / "mutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
                    "-D_GNU_SOURCE", "-o", str(so), str(c), "-lm"], check=True)
    check()                                   # the real oracle passes
    saved = oracle._lib
    oracle._lib = oracle._bind(ctypes.CDLL(str(so)))
    try:
        with pytest.raises(AssertionError):
            check()
    finally:
        oracle._lib = saved
