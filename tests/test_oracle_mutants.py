"""Planted mistakes in the oracle must be caught by its pins.

Each case copies oracle/kda_oracle.c, applies one textual mutation (a dropped
term, a wrong sign, index or operand), builds the copy into a temporary
directory and runs the whole pin battery against it in a child process (so a
crashing mutant cannot take the test run down).  The test passes when at least
one pin fails for every mutant.  Everything runs on the CPU.
"""
import json
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "kda_oracle.c")

DECAY = """                for (int c = 0; c < dk; ++c) {
                    const double a = exp(gt[c]);
                    for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] *= a;
                }
"""
UPDATE = """                for (int c = 0; c < dk; ++c) {
                    const double bk = bt * kt[c];
                    for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] += bk * (vt[j] - u[j]);
                }
"""

MUTANTS = {
    "beta_dropped_in_write": [("const double bk = bt * kt[c];", "const double bk = kt[c];")],
    "erase_sign_flipped": [("+= bk * (vt[j] - u[j]);", "+= bk * (vt[j] + u[j]);")],
    "decay_inverted": [("const double a = exp(gt[c]);", "const double a = exp(-gt[c]);")],
    "decay_after_erase": [(DECAY + "                for (int j = 0; j < dv; ++j) u[j] = 0.0;\n",
                           "                for (int j = 0; j < dv; ++j) u[j] = 0.0;\n"),
                          (UPDATE, UPDATE + DECAY)],
    "read_with_key": [("u[j] += S[(size_t)c * dv + j] * qt[c];", "u[j] += S[(size_t)c * dv + j] * kt[c];")],
    "scale_dropped": [("double r = scale * u[j];", "double r = u[j];")],
    "gate_without_sigmoid": [("double r = scale * u[j];\n                    if (gate) r *= sigm(",
                              "double r = scale * u[j];\n                    if (gate) r *= (")],
    "conv_tap_shifted": [("long tau = t - R + i;", "long tau = t - R + i - 1;")],
    "conv_without_silu": [("y[(s + t) * D + c] = apply_silu ? acc * sigm(acc) : acc;", "y[(s + t) * D + c] = acc;")],
    "conv_state_reversed": [("cs_out[((size_t)n * R + r) * D + c] = xv;",
                             "cs_out[((size_t)n * R + (R - 1 - r)) * D + c] = xv;")],
    "l2_eps_outside_root": [("double inv = 1.0 / sqrt(ss + eps);", "double inv = 1.0 / (sqrt(ss) + eps);")],
    "l2_missing_root": [("double inv = 1.0 / sqrt(ss + eps);", "double inv = 1.0 / (ss + eps);")],
    "backward_drops_key_path_through_u": [("gk[tk + c] = bt * (gu - ph);", "gk[tk + c] = bt * gu;")],
    "backward_skips_decay": [("G[(size_t)c * dv + j] = al * dP;", "G[(size_t)c * dv + j] = dP;")],
    "backward_misses_output_term": [("G[(size_t)c * dv + j] += scale * qt[c] * dOt[j];",
                                     "G[(size_t)c * dv + j] += 0.0 * qt[c] * dOt[j];")],
    "backward_reads_old_state_for_q": [("a += St[(size_t)c * dv + j] * dOt[j];", "a += Sp[(size_t)c * dv + j] * dOt[j];")],
    "state_not_reset_between_sequences": [
        ("for (long t = cu[n]; t < cu[n + 1]; ++t) {\n                const double *qt = q + ((size_t)t * H + h) * dk;\n                const double *kt = k + ((size_t)t * H + h) * dk;\n                const double *gt = g + ((size_t)t * H + h) * dk;\n                const double *vt = v + ((size_t)t * H + h) * dv;\n                const double bt = beta[(size_t)t * H + h];\n                for (int c = 0; c < dk; ++c) {\n                    const double a",
         "for (long t = (cu[n] > 0 ? cu[n] - 1 : 0); t < cu[n + 1]; ++t) {\n                const double *qt = q + ((size_t)t * H + h) * dk;\n                const double *kt = k + ((size_t)t * H + h) * dk;\n                const double *gt = g + ((size_t)t * H + h) * dk;\n                const double *vt = v + ((size_t)t * H + h) * dv;\n                const double bt = beta[(size_t)t * H + h];\n                for (int c = 0; c < dk; ++c) {\n                    const double a")],
}

RUNNER = """
import json, sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import oracle, oracle_pins
lib = oracle.load({lib!r})
print(json.dumps(oracle_pins.failing_pins(lib)))
"""


def _mutate(text, edits):
    for old, new in edits:
        assert text.count(old) == 1, f"mutation anchor not unique/present: {old[:60]!r}"
        text = text.replace(old, new)
    return text


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    with open(SRC) as f:
        src = _mutate(f.read(), MUTANTS[name])
    msrc = tmp_path / "mutant.c"
    msrc.write_text(src)
    lib = oracle.build(force=True, out_path=str(tmp_path / "libmutant.so"), src=str(msrc))
    code = RUNNER.format(root=ROOT, tests=os.path.join(ROOT, "tests"), lib=lib)
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    if res.returncode != 0:
        return                                   # the mutant crashed the pin run: caught
    failed = json.loads(res.stdout.strip().splitlines()[-1])
    assert failed, f"mutant {name} passed every pin"


def test_unmutated_oracle_passes_all_pins(tmp_path):
    lib = oracle.build(force=True, out_path=str(tmp_path / "libclean.so"))
    code = RUNNER.format(root=ROOT, tests=os.path.join(ROOT, "tests"), lib=lib)
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr
    assert json.loads(res.stdout.strip().splitlines()[-1]) == []
