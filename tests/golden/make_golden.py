"""Writes the stored oracle fixtures under tests/golden/ (calls only oracle/).

The pages print no worked numeric example, so these fixtures hold no page
values: each is a small seeded case run through the fp64 token loop (the
per-token recurrence of the "Kimi K3" blog, section "Kimi Delta Attention"),
with its inputs stored next to the outputs.  They record what the oracle
computed when it was pinned, so that a later change to its arithmetic, or a
build on another host (compiler, architecture, OpenMP thread count), shows up
as a mismatch in tests/test_golden.py instead of passing silently.

    python tests/golden/make_golden.py
"""
from __future__ import annotations

import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402

CASES = {
    # two sequences (ragged, one shorter than anything a chunk would hold) and
    # an empty one; random S0; 2 heads; d_k = 4, d_v = 3
    "oracle_varlen_T23_H2_dk4_dv3": dict(seed=1, lengths=[17, 0, 6], H=2, dk=4, dv=3),
}


def make(seed, lengths, H, dk, dv):
    rng = np.random.default_rng(seed)
    T = sum(lengths)
    f32 = lambda x: x.astype(np.float32).astype(np.float64)
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q, k = f32(q), f32(k)
    v = f32(rng.standard_normal((T, H, dv)))
    log_alpha = f32(np.clip(-np.log1p(np.exp(rng.standard_normal((T, H, dk)))), -5.0, -1e-4))
    beta = f32(1.0 / (1.0 + np.exp(-rng.standard_normal((T, H)))))
    S0 = 0.1 * rng.standard_normal((len(lengths), H, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    O, Sf = oracle.prefill(q, k, v, log_alpha, beta, cu_seqlens=cu, S0=S0)
    return dict(cu_seqlens=cu.tolist(), q=q.tolist(), k=k.tolist(), v=v.tolist(), log_alpha=log_alpha.tolist(),
                beta=beta.tolist(), S0=S0.tolist(), O=O.tolist(), S_final=Sf.tolist())


def main():
    for name, spec in CASES.items():
        data = dict(source="oracle.prefill (fp64 token loop), written by tests/golden/make_golden.py",
                    spec=spec, **make(**spec))
        with open(os.path.join(HERE, name + ".json"), "w") as f:
            json.dump(data, f, indent=None, separators=(",", ":"))
            f.write("\n")
        print("wrote", name)


if __name__ == "__main__":
    main()
