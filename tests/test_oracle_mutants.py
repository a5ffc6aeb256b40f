"""The pins must catch plausible mistakes in the oracle.

Each case below plants one mistake in a copy of ``oracle/sv_oracle.c`` (a
flipped sign, a swapped operand, a wrong index, a dropped term...), builds the
copy into a temporary directory and runs the pin suite against it in a fresh
process. The suite has to fail for every one of them. Nothing here touches the
real oracle or any GPU.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "sv_oracle.c")

MUTANTS = {
    "residual_sign_flipped": ("w[k] = (p > q) ? (p - q) : 0.0;", "w[k] = (q > p) ? (q - p) : 0.0;"),
    "ratio_inverted": ("return exp(log_p - log_q);", "return exp(log_q - log_p);"),
    "accept_test_inverted": ("if (!(u < r)) {", "if (u < r) {"),
    "no_truncation": ("            j = i;\n            break;\n        }\n    }\n\n    /* Step 3",
                      "            j = i;\n        }\n    }\n\n    /* Step 3"),
    "bonus_row_off_by_one": ("filtered_weights(trow0 + (size_t)K * V * esz, NULL",
                             "filtered_weights(trow0 + (size_t)(K - 1) * V * esz, NULL"),
    "race_score_inverted": ("double score = w / (-log(v));", "double score = w * (-log(v));"),
    "race_clock_sign": ("double score = w / (-log(v));", "double score = w / log(v);"),
    "race_lane_fixed": ("(2u * (r[k & 3u] >> 9) + 1u)", "(2u * (r[0] >> 9) + 1u)"),
    "race_shares_accept_counter": ("ctr[2] = 1u + (k >> 2); ctr[3] = 0;",
                                   "ctr[2] = (k >> 2); ctr[3] = 0;"),
    "block_race_shares_token_stream": ("ctr[2] = 1u + (c >> 2); ctr[3] = 1;",
                                       "ctr[2] = 1u + (c >> 2); ctr[3] = 0;"),
    "block_weight_ignored": ("if (W > 0.0) race_step(W,", "if (W > 0.0) race_step(1.0,"),
    "level2_races_wrong_block": ("k0 = best_c * block;", "k0 = 0;"),
    "level2_block_start_shifted": ("k0 = best_c * block;", "k0 = best_c * block + 1;"),
    "block_weight_skips_first_token": ("for (k = k0; k < k1; ++k) W += w[k];",
                                       "for (k = k0 + 1; k < k1; ++k) W += w[k];"),
    "block_length_fixed": ("nblocks = (V + block - 1) / block;",
                           "block = 512;\n    nblocks = (V + block - 1) / block;"),
    "temperature_dropped_in_max": ("double s = svo_elem(row, k, dtype) / T;",
                                   "double s = svo_elem(row, k, dtype);"),
    "lse_shift_sign": ("acc += exp(svo_elem(row, k, dtype) / T - m);",
                       "acc += exp(svo_elem(row, k, dtype) / T + m);"),
    "argmax_last_occurrence": ("else if (v > best) {", "else if (v >= best) {"),
    "philox_words_swapped": ("uint32_t y1 = lo1;", "uint32_t y1 = lo0;"),
    "philox_key_schedule_dropped": ("k1 += PHILOX_W1;", ""),
    "draft_row_index": ("thr[K + 1 + i], lm[K + 1 + i]);\n        /* A token",
                        "thr[K + 1 + i], lm[K + 1 + i]);\n        lq = filtered_log_prob(drow0, x, dtype, T, lse_d[0], thr[K + 1], lm[K + 1]);\n        /* A token"),
    "uniform_shift": ("(r[lane & 3] >> 8)", "(r[lane & 3] >> 9)"),
    "topk_rank_off_by_one": ("thr_k = v[top_k - 1];", "thr_k = v[top_k];"),
    "topp_target_ignores_topk_mass": ("const double target = top_p * mass_k;",
                                      "const double target = top_p;"),
    "topp_ties_split": ("g < V && v[g] == v[k]; ++g)", "g < V && g == k; ++g)"),
    "topp_keeps_one_group_less": ("*thr = v[k] > thr_k ? v[k] : thr_k;",
                                  "*thr = (k > 0 ? v[k - 1] : v[k]) > thr_k ? (k > 0 ? v[k - 1] : v[k]) : thr_k;"),
    "filtered_mass_not_renormalised": ("return svo_log_prob(row, k, dtype, T, lse) - log_mass;",
                                       "return svo_log_prob(row, k, dtype, T, lse);"),
    "draft_left_unfiltered": ("&thr[K + 1 + i], &lm[K + 1 + i], &mg);",
                              "&mg, &mg, &mg);"),
    "zero_target_mass_accepted": ("double r = lp == -INFINITY ? 0.0 : svo_accept_prob(lp, lq);",
                                  "double r = svo_accept_prob(lp, lq);"),
    "bonus_row_unfiltered": ("lse_t[K], thr[K], lm[K],", "lse_t[K], -INFINITY, 0.0,"),
    "f64_reader_stride": ("memcpy(&d, (const unsigned char*)row + 8 * k, 8);",
                          "memcpy(&d, (const unsigned char*)row + 4 * k, 8);"),
    "f64_read_as_f32": ("    if (dtype == SVO_F64) {\n        double d;",
                        "    if (dtype == -1) {\n        double d;"),
}


@pytest.mark.slow
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutant = tmp_path / "sv_oracle.c"
    mutant.write_text(src.replace(old, new))
    (tmp_path / "sv_oracle.h").write_text(open(os.path.join(ROOT, "oracle", "sv_oracle.h")).read())
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-o", str(so), str(mutant),
                    "-lm"], check=True)
    env = dict(os.environ, SVO_LIB_PATH=str(so))
    p = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_lmhead.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert p.returncode != 0, f"mutant {name} passed every pin:\n{p.stdout[-2000:]}"
    assert "failed" in p.stdout, p.stdout[-2000:]
