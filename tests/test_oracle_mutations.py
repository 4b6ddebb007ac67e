"""The pins catch plausible mistakes: each case plants one mistake in a copy of
ssu_oracle.c (on the CPU), builds it, and runs the pin suites against it; at
least one pin must fail."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ssu_oracle.c")

MUTANTS = {
    "decay_after_input": ("*hv = *hv * dA + dt * xp * Bn;", "*hv = (*hv + dt * xp * Bn) * dA;"),
    "input_without_dt": ("*hv = *hv * dA + dt * xp * Bn;", "*hv = *hv * dA + xp * Bn;"),
    "y_from_old_state": ("      *hv = *hv * dA + dt * xp * Bn;\n      acc += *hv * Cn;",
                         "      acc += *hv * Cn;\n      *hv = *hv * dA + dt * xp * Bn;"),
    "dropped_D": ("double out = acc + D * xp;", "double out = acc;"),
    "B_C_swapped": ("const double Bn = load_value(o->B,", "const double Bn = load_value(o->C,"),
    "interleaved_groups": ("const int64_t g = h / (H / o->G);", "const int64_t g = h % o->G;"),
    "no_softplus": ("if (o->dt_softplus) dt = softplus(dt);", "(void)softplus;"),
    "bias_subtracted": ("dt += bias;", "dt -= bias;"),
    "sigmoid_gate": ("static double silu(double v) { return v / (1.0 + exp(-v)); }",
                     "static double silu(double v) { return 1.0 / (1.0 + exp(-v)); }"),
    "count_not_minus_one": ("num_accepted ? num_accepted[s] - 1 : 0", "num_accepted ? num_accepted[s] : 0"),
    "write_when_read_padded": ("const int write_ok = read_ok && !disable_state_update",
                               "const int write_ok = !disable_state_update"),
    "update_off_by_one": ("ring_start[slot] = must_checkpoint ? add_i32(start, prev) % ring_buffer_len : start;",
                          "ring_start[slot] = must_checkpoint ? add_i32(start, prev + 1) % ring_buffer_len : start;"),
    "update_ge_window": ("add_i32(prev, 1) > logical_window", "add_i32(prev, 1) >= logical_window"),
    "commit_branches_swapped": ("(must_checkpoint ? a : add_i32(acc, a))", "(must_checkpoint ? add_i32(acc, a) : a)"),
    "commit_ignores_pql": ("const int must_checkpoint = pql > 0 && add_i32(acc, pql)",
                           "const int must_checkpoint = add_i32(acc, pql)"),
    "channel_index_transposed": ("(o->param_per_dim & 1) ? o->A[h * P + p]",
                                 "(o->param_per_dim & 1) ? o->A[p * H + h]"),
    "bf16_truncates": ("double r = nearbyint(fabs(v) / quantum) * quantum;",
                       "double r = floor(fabs(v) / quantum) * quantum;"),
    # ReplaySSM
    "replay_checkpoint_at_window": ("const int checkpoint = ok && (int64_t)k + L > logical_window;",
                                    "const int checkpoint = ok && (int64_t)k + L >= logical_window;"),
    "replay_checkpoint_skipped": ("        if (checkpoint)\n", "        if (0 && checkpoint)\n"),
    "replay_new_position_without_k": ("const int64_t pos = ((int64_t)start + k + t) % ring_len;",
                                      "const int64_t pos = ((int64_t)start + t) % ring_len;"),
    "replay_one_token_short": ("        for (int32_t j = 0; j < k; ++j)\n          replay_token(",
                               "        for (int32_t j = 0; j + 1 < k; ++j)\n          replay_token("),
    "replay_ring_start_ignored": (
        "          replay_token(&o, h, x_cache, B_cache, dt_cache, slot, ((int64_t)start + j) % ring_len,",
        "          replay_token(&o, h, x_cache, B_cache, dt_cache, slot, ((int64_t)j) % ring_len,"),
    "replay_caches_biased_dt": ("dt_cache[(slot * H + h) * ring_len + pos] = dt[r * H + h];",
                                "dt_cache[(slot * H + h) * ring_len + pos] = dt[r * H + h] + "
                                "(dt_bias ? dt_bias[h] : 0.0f);"),
    "replay_B_of_first_group": ("B, (r * G + g) * N + n,", "B, (r * G + 0) * N + n,"),
    "replay_trackers_for_unprocessed": ("      if (!processed[s]) continue;\n",
                                        "      (void)processed;\n"),
    # stochastic rounding
    "sr_threshold_strict": ("frac >= 1.0 - ldexp((double)r, -16)",
                            "frac > 1.0 - ldexp((double)r, -16)"),
    "sr_counter_per_element": ("const uint64_t counter[4] = {(uint64_t)e >> 4, 0, 0, 0}",
                               "const uint64_t counter[4] = {(uint64_t)e, 0, 0, 0}"),
    "sr_word_from_low_bits": ("out[((uint64_t)e >> 2) & 3]", "out[(uint64_t)e & 3]"),
    "philox_weyl_swapped": ("k0 += 0x9E3779B97F4A7C15ull;", "k0 += 0xBB67AE8584CAA73Bull;"),
    "philox_halves_swapped": ("const uint64_t n0 = hi1 ^ x1 ^ k0, n1 = lo1, n2 = hi0 ^ x3 ^ k1, n3 = lo0;",
                              "const uint64_t n0 = lo1 ^ x1 ^ k0, n1 = hi1, n2 = hi0 ^ x3 ^ k1, n3 = lo0;"),
    "sr_ignored_in_state_writes": ("if (!sr || !sr->seed || (dtype != OR_BF16",
                                   "if (1 || !sr || !sr->seed || (dtype != OR_BF16"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutated = tmp_path / "ssu_oracle_mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o",
                    str(lib), str(mutated), "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_trackers.py"),
                        os.path.join(ROOT, "tests", "test_oracle_replay.py"),
                        os.path.join(ROOT, "tests", "test_oracle_sr.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
