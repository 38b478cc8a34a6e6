"""Planted mistakes: each pin of the oracle must be able to fail.

Every case below plants one plausible mistake in a copy of the oracle's C
source (a dropped term, a wrong sign, a step in the wrong order, a checkpoint
off by one segment), builds that copy, points the oracle wrapper at it and
runs the pins of tests/test_oracle_pins.py.  The case passes when at least
one pin rejects the mutant.  The unmodified source, built the same way, must
pass every pin (so a failure is the mistake's, not the harness's).

The mistakes are planted in the oracle only, on the CPU; nothing here touches
the CUDA library.
"""
import ctypes
import os
import subprocess

import pytest

import test_oracle_pins as pins
from oracle import oracle

SRC = oracle.SRC

# name -> [(exact text in kda_oracle.c, replacement)]
MUTANTS = {
    "beta missing from the correction": [
        ("e[j] = T->beta * ((real)vt[j] - s);", "e[j] = ((real)vt[j] - s);")],
    "output scale missing": [
        ("ot[j] = (double)(scale * s);", "ot[j] = (double)(s);")],
    "correction read from the undecayed state": [
        ("for (int i = 0; i < dk; i++) s += S[i * dv + j] * T->kh[i];",
         "for (int i = 0; i < dk; i++) s += S[i * dv + j] / (real)exp((double)T->g[i]) * T->kh[i];")],
    "softplus dropped from the gate": [
        ("T->g[i] = -a * sp_(T->x[i]);", "T->g[i] = -a * T->x[i];")],
    "L2-norm epsilon dropped": [
        ("T->nq = (real)sqrt((double)(sq + eps));", "T->nq = (real)sqrt((double)(sq));")],
    "decay missing from the state gradient": [
        ("dS[i * dv + j] *= al;", "")],
    "sign of the correction's gradient flipped": [
        ("du[j] = -T.beta * de[j];", "du[j] = T.beta * de[j];")],
    "output scale missing from the state gradient": [
        ("dS[i * dv + j] += (real)scale * T.qh[i] * (real)dot[j];",
         "dS[i * dv + j] += T.qh[i] * (real)dot[j];")],
    "L2-norm projection missing from dq": [
        ("(double)((dqh[i] - T.qh[i] * pq) / T.nq)", "(double)(dqh[i] / T.nq)")],
    "sigmoid derivative missing from db": [
        ("(double)(dbeta * T.beta * (1 - T.beta))", "(double)(dbeta)")],
    "dA_log term without g": [
        ("dAl += dg * T.g[i];", "dAl += dg;")],
    "checkpoint restored one segment late": [
        ("memcpy(seg, ckp + s * SS, sizeof(real) * SS);",
         "memcpy(seg, ckp + (s + 1 < nseg ? s + 1 : s) * SS, sizeof(real) * SS);")],
}

# the pins, called directly (float64 oracle)
PINS = [
    ("one step from zero", lambda: pins.test_one_step_from_zero_state("f64")),
    ("beta = 0 pure decay", lambda: pins.test_beta_zero_is_pure_decay("f64")),
    ("ungated delta rule", lambda: pins.test_ungated_delta_rule_orthonormal_keys("f64")),
    ("beta = 1 retrieval", lambda: pins.test_beta_one_write_is_retrievable("f64")),
    ("linearity", lambda: pins.test_linear_in_v_and_column_independent("f64")),
    ("dense transfer", lambda: pins.test_dense_transfer_products("f64")),
    ("chunked WY", lambda: pins.test_chunked_wy_form_matches(5)),
    ("finite differences", pins.test_finite_differences_every_gradient),
    ("finite differences across segments", pins.test_finite_differences_across_checkpoint_segments),
    ("large gates", pins.test_gradients_with_large_gates_and_no_h0),
    ("zero-length document", pins.test_zero_length_document_passes_state_through),
]


def _build(text, tmp_path, name):
    src = tmp_path / f"{name}.c"
    out = tmp_path / f"{name}.so"
    src.write_text(text)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                           "-DORACLE_REAL=double", "-o", str(out), str(src), "-lm"])
    return oracle.declare(ctypes.CDLL(str(out)))


def _failing_pins(lib, monkeypatch, stop_at_first):
    monkeypatch.setitem(oracle._libs, "f64", lib)
    failed = []
    for name, fn in PINS:
        try:
            fn()
        except AssertionError:
            failed.append(name)
            if stop_at_first:
                break
    return failed


def test_unmodified_source_passes_every_pin(tmp_path, monkeypatch):
    with open(SRC) as fh:
        lib = _build(fh.read(), tmp_path, "original")
    assert _failing_pins(lib, monkeypatch, stop_at_first=False) == []


@pytest.mark.parametrize("mutant", list(MUTANTS))
def test_planted_mistake_fails_a_pin(mutant, tmp_path, monkeypatch):
    with open(SRC) as fh:
        text = fh.read()
    for old, new in MUTANTS[mutant]:
        assert text.count(old) == 1, f"mutation site not unique: {old!r}"
        text = text.replace(old, new)
    lib = _build(text, tmp_path, "mutant")
    assert _failing_pins(lib, monkeypatch, stop_at_first=True), f"no pin rejects: {mutant}"
