"""Stored oracle fixtures (tests/golden/, written by tests/golden/make_golden.py
from the fp64 token loop) are reproduced by the oracle as built on this host,
and by the chunk form of the "Kimi K3: the manos, the mythos, the legendos"
page ("FlashKDA Algorithm") evaluated independently in numpy."""
import glob
import json
import os

import numpy as np
import pytest

import oracle
from oracle.chunked import prefill_chunked
from _pins import rel

GOLDEN = sorted(glob.glob(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "*.json")))


def load(path):
    d = json.load(open(path))
    arr = {key: np.asarray(d[key], dtype=np.float64) for key in ("q", "k", "v", "log_alpha", "beta", "S0", "O", "S_final")}
    arr["cu_seqlens"] = np.asarray(d["cu_seqlens"], dtype=np.int64)
    return d, arr


def test_fixtures_exist():
    assert GOLDEN, "no stored fixtures under tests/golden/"


@pytest.mark.parametrize("path", GOLDEN, ids=[os.path.basename(p) for p in GOLDEN])
@pytest.mark.parametrize("n_threads", [1, 3])
def test_oracle_reproduces_stored_fixture(path, n_threads):
    d, a = load(path)
    assert "oracle" in d["source"]
    O, Sf = oracle.prefill(a["q"], a["k"], a["v"], a["log_alpha"], a["beta"], cu_seqlens=a["cu_seqlens"],
                           S0=a["S0"], n_threads=n_threads)
    # the C loop's order of operations is fixed; only FMA contraction may differ between hosts
    assert rel(O, a["O"]) < 1e-12
    assert rel(Sf, a["S_final"]) < 1e-12


@pytest.mark.parametrize("path", GOLDEN, ids=[os.path.basename(p) for p in GOLDEN])
@pytest.mark.parametrize("chunk", [1, 4, 16])
def test_chunk_form_reproduces_stored_fixture(path, chunk):
    _, a = load(path)
    O, Sf = prefill_chunked(a["q"], a["k"], a["v"], a["log_alpha"], a["beta"], a["cu_seqlens"], chunk, S0=a["S0"])
    assert rel(O, a["O"]) < 1e-10
    assert rel(Sf, a["S_final"]) < 1e-10
