"""Planted mistakes in the oracle must trip the pins (CPU only).

Each mutant is a copy of ``oracle/kda_oracle.c`` with one plausible mistake
(a dropped term, a wrong sign, a transposed index, a reordered step), compiled
into a temporary directory.  The pin suite runs against it and at least one
pin has to fail; the unmodified oracle passes all of them (``test_oracle.py``).
"""

import os
import shutil
import subprocess

import pytest

import oracle
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")

# (name, text in the oracle, replacement)
MUTANTS = [
    ("gate_without_exp_on_A", "const double scale = exp(A[h]);", "const double scale = A[h];"),
    ("gate_wrong_sign", "g[i] = g_min / (1.0 + exp(-x));", "g[i] = g_min / (1.0 + exp(x));"),
    ("decay_sign_flipped", "const double alpha = exp(gt[c]);",
     "const double alpha = exp(-gt[c]);"),
    ("erase_reads_undecayed_state", "for (int j = 0; j < dv; ++j) kX[j] += kt[c] * X[c * dv + j];",
     "for (int j = 0; j < dv; ++j) kX[j] += kt[c] * S[c * dv + j];"),
    ("erase_without_beta",
     "S[c * dv + j] = X[c * dv + j] - bt * kt[c] * kX[j] + bt * kt[c] * vt[j];",
     "S[c * dv + j] = X[c * dv + j] - kt[c] * kX[j] + bt * kt[c] * vt[j];"),
    ("write_without_beta",
     "S[c * dv + j] = X[c * dv + j] - bt * kt[c] * kX[j] + bt * kt[c] * vt[j];",
     "S[c * dv + j] = X[c * dv + j] - bt * kt[c] * kX[j] + kt[c] * vt[j];"),
    ("h0_transposed", "J->h0[(((int64_t)n * H + h) * dv + j) * dk + c]",
     "J->h0[(((int64_t)n * H + h) * dk + c) * dv + j]"),
    ("readout_with_key", "acc += S[c * dv + j] * qt[c];", "acc += S[c * dv + j] * kt[c];"),
    ("readout_before_update_state", "for (int c = 0; c < dk; ++c) acc += S[c * dv + j] * qt[c];",
     "for (int c = 0; c < dk; ++c) acc += X[c * dv + j] * qt[c];"),
    ("state_not_reset_per_sequence", "S[c * dv + j] = J->h0 ? J->h0[",
     "S[c * dv + j] += J->h0 ? J->h0["),
]


def _decay_after_erase(src: str) -> str:
    """Apply the decay after the erase: S_t = D (I - b k k^T) S + b k v^T."""
    old = "for (int j = 0; j < dv; ++j) kX[j] += kt[c] * X[c * dv + j];"
    assert old in src
    src = src.replace(old, "for (int j = 0; j < dv; ++j) kX[j] += kt[c] * S[c * dv + j];")
    old2 = "S[c * dv + j] = X[c * dv + j] - bt * kt[c] * kX[j] + bt * kt[c] * vt[j];"
    assert old2 in src
    return src.replace(old2, "S[c * dv + j] = X[c * dv + j] - bt * kt[c] * kX[j] * exp(gt[c])"
                             " + bt * kt[c] * vt[j];")


def _build(tmp_path, name, text):
    d = tmp_path / name
    d.mkdir()
    src = d / "kda_oracle.c"
    src.write_text(text)
    out = str(d / "libkda_oracle.so")
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread", str(src),
                           "-o", out, "-lm"])
    return oracle.load(out)


def _tripped(lib):
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError, FloatingPointError):
            failed.append(pin.__name__)
    return failed


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert old in src, f"mutation anchor for {name} not found"
    lib = _build(tmp_path, name, src.replace(old, new, 1))
    assert _tripped(lib), f"no pin caught mutant {name}"


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_mutant_decay_after_erase_is_caught(tmp_path):
    lib = _build(tmp_path, "decay_after_erase", _decay_after_erase(open(SRC).read()))
    failed = _tripped(lib)
    assert "pin_delta_overwrite_any_decay" in failed or "pin_explicit_matrix_form" in failed
