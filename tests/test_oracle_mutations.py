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
                        os.path.join(ROOT, "tests", "test_oracle_trackers.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
