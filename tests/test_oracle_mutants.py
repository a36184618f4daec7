"""Plant mistakes in copies of the oracle's C source and check that the pins
catch every one of them (CPU only).  The mutants are built from the same
``kda_ref.c`` text with one substitution each; the oracle itself is untouched."""
import os
import shutil
import subprocess

import pytest

import oracle
from _pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_ref.c")

MUTANTS = {
    "delta_sign": ("x[j] = bt * ((double)vt[j] - x[j]);", "x[j] = bt * ((double)vt[j] + x[j]);"),
    "no_decay": ("for (int j = 0; j < dv; ++j) Si[j] *= a;", "for (int j = 0; j < dv; ++j) Si[j] *= 1.0;"),
    "base2_gate": ("const double a = exp((double)gt[i]);", "const double a = exp2((double)gt[i]);"),
    "beta_dropped": ("x[j] = bt * ((double)vt[j] - x[j]);", "x[j] = 1.0 * ((double)vt[j] - x[j]);"),
    "readout_uses_k": ("const double qi = (double)qt[i];", "const double qi = (double)kt[i];"),
    "first_token_skipped": ("for (int64_t t = bos; t < eos; ++t) {", "for (int64_t t = bos + 1; t < eos; ++t) {"),
    "s0_ignored": ("if (S0_nh)\n", "if (0)\n"),
    "gate_on_columns": ("for (int j = 0; j < dv; ++j) Si[j] *= a;",
                        "for (int j = 0; j < dv; ++j) Si[j] *= exp((double)gt[j]);"),
    "beta_squared": ("x[j] = bt * ((double)vt[j] - x[j]);", "x[j] = bt * bt * ((double)vt[j] - x[j]);"),
    "state_carried_across_sequences": ("    else\n        memset(S, 0, sizeof(double) * (size_t)dk * dv);",
                                       "    else if (bos == 0)\n        memset(S, 0, sizeof(double) * (size_t)dk * dv);"),
    "readout_before_write": (
        "        /* Delta-rule write: S += k_t (beta_t (v_t - v_old))^T. */",
        "        if (O) {\n            double* ot = O + ((size_t)t * Hs + hs) * dv;\n"
        "            for (int j = 0; j < dv; ++j) ot[j] = 0.0;\n"
        "            for (int i = 0; i < dk; ++i) for (int j = 0; j < dv; ++j) ot[j] += S[(size_t)i*dv+j] * qt[i];\n"
        "        }\n"
        "        /* Delta-rule write: S += k_t (beta_t (v_t - v_old))^T. */"),
    "vold_before_decay": (
        "        /* Decay old memory: row i of S times alpha_t[i]. */",
        "        for (int j = 0; j < dv; ++j) x[j] = 0.0;\n"
        "        for (int i = 0; i < dk; ++i) for (int j = 0; j < dv; ++j) x[j] += S[(size_t)i*dv+j] * (double)kt[i];\n"
        "        /* Decay old memory: row i of S times alpha_t[i]. */"),
}


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation anchor for {name} not found"
    if name == "readout_before_write":
        # read out from the decayed state before the write; the read-out after the write is dropped
        text = text.replace(old, new, 1)
        text = text.replace("        /* Read-out o_t = S_t^T q_t (after the write). */\n        if (O) {",
                            "        /* Read-out o_t = S_t^T q_t (after the write). */\n        if (0) {", 1)
    elif name == "vold_before_decay":
        # compute v_old from the undecayed state, then skip the later v_old pass
        text = text.replace(old, new, 1)
        text = text.replace("        /* v_old = Sbar^T k_t. */\n        for (int j = 0; j < dv; ++j) x[j] = 0.0;\n"
                            "        for (int i = 0; i < dk; ++i) {\n            const double ki = (double)kt[i];\n"
                            "            const double* Si = S + (size_t)i * dv;\n"
                            "            for (int j = 0; j < dv; ++j) x[j] += Si[j] * ki;\n        }\n", "", 1)
    else:
        text = text.replace(old, new, 1)
    src = tmp_path / f"{name}.c"
    src.write_text(text)
    lib = oracle.bind(oracle.compile_source(str(src), str(tmp_path / f"lib{name}.so")))
    run = lambda *a, **kw: oracle.prefill(*a, lib=lib, **kw)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(run)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {name}"


# Mistakes in the fused prologue, caught by the prologue's own pins
# (tests/test_oracle_prologue.py), run against the mutant build.
PROLOGUE_MUTANTS = {
    "eps_outside_sqrt": ("return 1.0 / sqrt(ss + 1e-6);", "return 1.0 / (sqrt(ss) + 1e-6);"),
    "softplus_sign": ("const double lg = -log1p(exp(a));", "const double lg = -log1p(exp(-a));"),
    "no_lower_clamp": ("return lg < -5.0 ? -5.0 :", "return lg < -50.0 ? -50.0 :"),
    "sigmoid_sign": ("return 1.0 / (1.0 + exp(-b));", "return 1.0 / (1.0 + exp(b));"),
    "k_scaled_by_q_norm": ("const double ks = prologue ? prologue_unit_scale(k32, dk) : 1.0;",
                           "const double ks = prologue ? prologue_unit_scale(q32, dk) : 1.0;"),
    "gate_not_activated": ("gt[i] = prologue ? prologue_log_alpha((double)g32[i]) : (double)g32[i];",
                           "gt[i] = (double)g32[i];"),
}


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(PROLOGUE_MUTANTS))
def test_prologue_pins_catch_mutant(name, tmp_path, monkeypatch):
    import test_oracle_prologue as pp
    old, new = PROLOGUE_MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor for {name} not found"
    src = tmp_path / f"{name}.c"
    src.write_text(text.replace(old, new, 1))
    lib = oracle.bind(oracle.compile_source(str(src), str(tmp_path / f"lib{name}.so")))
    monkeypatch.setattr(oracle, "_load", lambda: lib)
    pins = [getattr(pp, n) for n in dir(pp) if n.startswith("test_")]
    caught = []
    for pin in pins:
        try:
            pin()
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no prologue pin caught mutant {name}"


def test_prologue_pins_pass_on_the_oracle():
    """The same loop over the unmodified oracle raises nothing (the mutant test
    above is not vacuous)."""
    import test_oracle_prologue as pp
    for n in dir(pp):
        if n.startswith("test_"):
            getattr(pp, n)()
