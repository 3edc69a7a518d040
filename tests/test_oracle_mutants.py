"""Planted mistakes in the oracle must be caught by its pins (CPU only).

Each case copies ``oracle/attention_oracle.c``, makes one plausible mistake in
the copy (a dropped term, a wrong sign, a wrong index, a transposed operand, a
wrong mask), compiles it to a temporary shared object and runs the pin checks
on it.  The case passes when at least one pin fails on the mutant.  The real
oracle source is never modified.
"""
import pytest

import oracle
from oracle_pin_checks import ALL_CHECKS

MUTANTS = {
    # forward
    "max_wrong_direction": ("if (s > m) m = s;", "if (s < m) m = s;"),
    "scale_dropped": ("return scale * acc;", "return acc;"),
    "lse_sign": ("lse[(long)h * Nq + i] = m + log(l);", "lse[(long)h * Nq + i] = m - log(l);"),
    "lse_log_dropped": ("lse[(long)h * Nq + i] = m + log(l);", "lse[(long)h * Nq + i] = m + l;"),
    "value_row_index": ("const double *vj = vh + j * d;", "const double *vj = vh + i * d;"),
    "causal_off_by_one": ("if (mk->causal && j > i + mk->off) return 0;",
                          "if (mk->causal && j >= i + mk->off) return 0;"),
    "causal_transposed": ("if (mk->causal && j > i + mk->off) return 0;",
                          "if (mk->causal && j < i + mk->off) return 0;"),
    "normaliser_dropped": (
        "double p = exp(score(qh + (long)i * d, kh + j * d, d, scale) - m) / l;",
        "double p = exp(score(qh + (long)i * d, kh + j * d, d, scale) - m);"),
    # backward
    "ds_D_sign": ("double ds = p * (dp - Di);", "double ds = p * (dp + Di);"),
    "ds_D_dropped": ("double ds = p * (dp - Di);", "double ds = p * dp;"),
    "dk_scale_dropped": ("dkj[c] += scale * ds * qh[i * d + c];", "dkj[c] += ds * qh[i * d + c];"),
    "dv_transposed": ("dvj[c] += p * dOh[i * d + c];", "dvj[c] += p * dOh[(long)j * d + c];"),
    "dq_wrong_operand": ("dqi[c] += scale * ds * kh[j * d + c];",
                         "dqi[c] += scale * ds * qh[j * d + c];"),
    "dp_transposed_in_key_pass": (
        "dp += dOh[i * d + c] * vh[(long)j * d + c];",
        "dp += dOh[(long)j * d + c] * vh[i * d + c];"),
    "key_pass_D_dropped": ("double ds = p * (dp - D[r]);", "double ds = p * dp;"),
    # the backward rows entry
    "bwd_rows_dk_wrong_operand": ("dkj[c] += scale * ds * q[i * d + c];",
                                  "dkj[c] += scale * ds * k[j * d + c];"),
    "bwd_rows_D_dropped": ("double ds = p * (dp - D[i]);", "double ds = p * dp;"),
    "bwd_rows_query_index": ("const long i = qrows[t];", "const long i = t;"),
    "bwd_rows_stats_top_left": ("if (visible(mk, i, krows[t])) need[i] = 1;",
                                "if (krows[t] <= i) need[i] = 1;"),
    # grouped key/value heads
    "gqa_kv_head_modulo": ("*kh = k + (h / group) * hk, *vh = v + (h / group) * hk;",
                           "*kh = k + (h % group) * hk, *vh = v + (h % group) * hk;"),
    "gqa_group_sum_first_head_only": ("for (int g = 0; g < group; ++g) {",
                                      "for (int g = 0; g < 1; ++g) {"),
    "gqa_interleaved_grouping": ("const int h = kv * group + g;", "const int h = g * BHkv + kv;"),
    # query and key lengths that differ
    "cross_causal_offset_dropped": ("if (mk->causal && j > i + mk->off) return 0;",
                                    "if (mk->causal && j > i) return 0;"),
    "cross_causal_offset_sign": ("if (mk->causal && j > i + mk->off) return 0;",
                                 "if (mk->causal && j > i - mk->off) return 0;"),
    "cross_offset_top_left": ("Mask mk = {causal, (long)Nk - Nq,", "Mask mk = {causal, 0,"),
    "cross_key_stride_query_len": ("hk = (long)Nk * d;", "hk = (long)Nq * d;"),
    "cross_key_loop_query_len": ("for (long j = 0; j < Nk; ++j) {\n                if (!visible(mk, i, j)) continue;\n                double p",
                                 "for (long j = 0; j < Nq; ++j) {\n                if (!visible(mk, i, j)) continue;\n                double p"),
    # block-sparse masks (the first block-sparse pin keeps these in bounds)
    "sparse_mask_inverted": ("mk->bm[(i / mk->bq) * (long)mk->nbk + j / mk->bk] != 0;",
                             "mk->bm[(i / mk->bq) * (long)mk->nbk + j / mk->bk] == 0;"),
    "sparse_mask_ignored_when_causal": ("return !mk->bm ||", "return mk->causal || !mk->bm ||"),
    "sparse_row_block_from_key_size": ("mk->bm[(i / mk->bq) *", "mk->bm[(i / mk->bk) *"),
    "sparse_row_stride_from_queries": ("bm ? (Nk + bk - 1) / bk : 0", "bm ? (Nq + bq - 1) / bq : 0"),
    "sparse_key_pass_ignores_mask": (
        "                    if (!visible(mk, i, j)) continue;",
        "                    if (mk->causal && j > i + mk->off) continue;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new)
    c_path = tmp_path / f"mutant_{name}.c"
    c_path.write_text(mutated)
    lib = oracle.OracleLib(oracle.compile_c(str(c_path), str(tmp_path / f"mutant_{name}.so")))
    failed = []
    for check in ALL_CHECKS:
        try:
            check(lib)
        except AssertionError:
            failed.append(check.__name__)
            break
    assert failed, f"no pin caught the planted mistake {name}"
