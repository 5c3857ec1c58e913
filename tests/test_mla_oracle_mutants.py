"""Planted mistakes in the MLA decode oracle must be caught by its pins.

Each case copies oracle/mla_oracle.c, applies one textual mutation, builds the
copy into a temporary directory and runs the MLA pin battery against it in a
child process.  The test passes when at least one pin fails for every mutant.
Everything runs on the CPU.
"""
import json
import os
import subprocess
import sys

import pytest

import oracle.mla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "mla_oracle.c")

MUTANTS = {
    "rope_sin_sign_flipped": [("x[i] = a * c - b * s;", "x[i] = a * c + b * s;"),
                              ("x[i + half] = b * c + a * s;", "x[i + half] = b * c - a * s;")],
    "rope_frequency_exponent": [("pow(theta, -2.0 * i / rd)", "pow(theta, -1.0 * i / rd)")],
    "rope_pairs_adjacent_dims": [("const double a = x[i], b = x[i + half];", "const double a = x[i], b = x[i ^ 1];")],
    "query_rotated_one_ahead": [("rope_row(qr, rd, pos, theta);", "rope_row(qr, rd, pos + 1, theta);")],
    "new_key_not_attended": [("for (int t = 0; t <= pos; ++t) {\n                double s = 0.0;",
                              "for (int t = 0; t < pos; ++t) {\n                double s = 0.0;")],
    "scale_dropped": [("sc[t] = scale * s;", "sc[t] = s;")],
    "softmax_not_normalised": [("double r = acc / den;", "double r = acc;")],
    "gate_without_sigmoid": [("if (gate) r *= 1.0 / (1.0 + exp(-gate[nh * dv + j]));",
                              "if (gate) r *= gate[nh * dv + j];")],
    "value_not_rounded_to_bf16": [("cache_bf16 ? round_bf16(v_new[nh * dv + j]) : v_new[nh * dv + j]",
                                   "v_new[nh * dv + j]")],
    "bf16_ties_away_from_zero": [("double r = nearbyint(s);", "double r = round(s);")],
    "length_not_advanced": [("if (valid) cache_len[n] = pos + 1;", "if (valid) cache_len[n] = pos;")],
    "full_cache_gives_zeros": [("for (int j = 0; j < dv; ++j) o[j] = NAN;", "for (int j = 0; j < dv; ++j) o[j] = 0.0;")],
}

RUNNER = """
import json, sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import oracle.mla, mla_oracle_pins
lib = oracle.mla.load({lib!r})
print(json.dumps(mla_oracle_pins.failing_pins(lib)))
"""


def _mutate(text, edits):
    for old, new in edits:
        assert text.count(old) == 1, f"mutation anchor not unique/present: {old[:60]!r}"
        text = text.replace(old, new)
    return text


def _run(lib):
    code = RUNNER.format(root=ROOT, tests=os.path.join(ROOT, "tests"), lib=lib)
    return subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    with open(SRC) as f:
        src = _mutate(f.read(), MUTANTS[name])
    msrc = tmp_path / "mutant.c"
    msrc.write_text(src)
    res = _run(oracle.mla.build(force=True, out_path=str(tmp_path / "libmutant.so"), src=str(msrc)))
    if res.returncode != 0:
        return                                   # the mutant crashed the pin run: caught
    failed = json.loads(res.stdout.strip().splitlines()[-1])
    assert failed, f"mutant {name} passed every pin"


def test_unmutated_oracle_passes_all_pins(tmp_path):
    res = _run(oracle.mla.build(force=True, out_path=str(tmp_path / "libclean.so")))
    assert res.returncode == 0, res.stderr
    assert json.loads(res.stdout.strip().splitlines()[-1]) == []
