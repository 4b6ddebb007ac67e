"""The SSD oracle's pins catch plausible mistakes: each case plants one mistake
in a copy of oracle/ssd.py (on the CPU) and runs tests/test_oracle_ssd.py
against it; at least one pin must fail."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ssd.py")

MUTANTS = {
    "clamp_before_softplus": (
        "            if dt_softplus:\n                d = softplus(d)\n"
        "            d = np.minimum(np.maximum(d, lo), hi)\n",
        "            d = np.minimum(np.maximum(d, lo), hi)\n"
        "            if dt_softplus:\n                d = softplus(d)\n"),
    "y_from_old_state": (
        "            h = h * dA[:, None, None] + (d[:, None] * x[t])[:, :, None] * Bt[:, None, :]\n"
        "            y = np.einsum(\"hpn,hn->hp\", h, Ct)\n",
        "            y = np.einsum(\"hpn,hn->hp\", h, Ct)\n"
        "            h = h * dA[:, None, None] + (d[:, None] * x[t])[:, :, None] * Bt[:, None, :]\n"),
    "decay_after_input": (
        "h = h * dA[:, None, None] + (d[:, None] * x[t])[:, :, None] * Bt[:, None, :]",
        "h = (h + (d[:, None] * x[t])[:, :, None] * Bt[:, None, :]) * dA[:, None, None]"),
    "chunks_never_open_a_sequence": ("if c == 0 or seq[c] != seq[c - 1]:", "if c == 0:"),
    "input_without_dt": ("(d[:, None] * x[t])[:, :, None]", "x[t][:, :, None]"),
    "last_chunk_off_by_one": ("states[last])", "states[np.maximum(last - 1, 0)])"),
    "interleaved_groups": ("group = np.arange(H) // (H // G)", "group = np.arange(H) % G"),
    "no_gate": ("y = y * (z[t] / (1.0 + np.exp(-z[t])))", "y = y"),
    "bias_subtracted": ("d = dt[t] + (dt_bias if dt_bias is not None else 0.0)",
                        "d = dt[t] - (dt_bias if dt_bias is not None else 0.0)"),
    "decay_without_dt": ("dA = np.exp(A * d)", "dA = np.exp(A)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutated = tmp_path / "ssd_mutant.py"
    mutated.write_text(src.replace(old, new))
    env = dict(os.environ, SSD_ORACLE_PATH=str(mutated))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_ssd.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
