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
    if name == "vold_before_decay":
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
