"""Pins of the fp64 oracle to facts the pages and the mathematics fix.

Each ``pin_*`` takes ``run`` -- a callable with the signature of
``oracle.prefill`` -- and raises AssertionError when the oracle disagrees with
the fact.  The facts come from outside the oracle's own code:

P1  the product form S_t = (I - b k k^T) Diag(a) S + b k v^T equals the
    two-stage form the oracle implements ("Kimi K3" blog, section "Kimi Delta
    Attention": the recurrent form and its "Decay Old Memory" / "Apply
    Delta-Rule Update" reading);
P2  beta = 0 means nothing is written: with alpha = 1 the state stays S0 and
    o_t = S0^T q_t; with a general gate S_T = Diag(prod alpha) S0;
P3  a gate that is equal on every key channel is Gated DeltaNet's scalar gate
    update S_t = a_t (I - b k k^T) S + b k v^T (same blog, Gated DeltaNet);
P4  beta = 1 and a unit key make the write exact: S_t^T k_t = v_t (the
    delta rule replaces v_old by v_t; "Apply Delta-Rule Update");
P5  the chunked matrix form ("Kimi K3: the manos, the mythos, the legendos",
    section "FlashKDA Algorithm") equals the token loop for every chunk size;
P6  orthonormal keys with beta = 1 and no decay turn S into a lookup table whose
    row i holds the last value written under key e_i;
P7  splitting a sequence and carrying the state equals one run; a packed
    varlen batch equals separate runs, with per-sequence S0 and without one
    (each sequence then starts from zero; the chunk unrolling holds from any
    starting state).
"""
from __future__ import annotations

import numpy as np

import oracle


def rand_inputs(rng, T, H, dk, dv, unit_k=True):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    if unit_k:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    g = -np.log1p(np.exp(rng.standard_normal((T, H, dk))))
    g = np.clip(g, -5.0, -1e-4)
    # round through fp32 so both sides see exactly the values the oracle reads
    return tuple(x.astype(np.float32).astype(np.float64) for x in (q, k, v, g, beta))


def product_form(q, k, v, g, beta, S0=None):
    """S_t = (I - b_t k_t k_t^T) Diag(alpha_t) S_{t-1} + b_t k_t v_t^T, o_t = S_t^T q_t."""
    T, H, dk = q.shape
    dv = v.shape[2]
    O = np.zeros((T, H, dv))
    Sf = np.zeros((H, dk, dv))
    for h in range(H):
        S = np.zeros((dk, dv)) if S0 is None else S0[h].copy()
        for t in range(T):
            kt = k[t, h][:, None]
            A = (np.eye(dk) - beta[t, h] * kt @ kt.T) @ np.diag(np.exp(g[t, h]))
            S = A @ S + beta[t, h] * kt @ v[t, h][None, :]
            O[t, h] = S.T @ q[t, h]
        Sf[h] = S
    return O, Sf


def rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def pin_p1_product_form(run, seed=1):
    rng = np.random.default_rng(seed)
    q, k, v, g, b = rand_inputs(rng, 9, 2, 6, 5, unit_k=False)
    S0 = rng.standard_normal((1, 2, 6, 5))
    O, Sf = run(q, k, v, g, b, S0=S0)
    Oe, Sfe = product_form(q, k, v, g, b, S0=S0[0])
    assert rel(O, Oe) < 1e-12, rel(O, Oe)
    assert rel(Sf[0], Sfe) < 1e-12, rel(Sf[0], Sfe)


def pin_p2_no_write(run, seed=2):
    rng = np.random.default_rng(seed)
    q, k, v, g, b = rand_inputs(rng, 11, 2, 4, 3)
    S0 = rng.standard_normal((1, 2, 4, 3))
    zero_b = np.zeros_like(b)
    # alpha = 1, beta = 0: plain read-out of a frozen state
    O, Sf = run(q, k, v, np.zeros_like(g), zero_b, S0=S0)
    assert np.array_equal(Sf[0], S0[0])
    Oe = np.einsum("thi,hij->thj", q, S0[0])
    assert rel(O, Oe) < 1e-14
    # beta = 0, general gate: only the decay acts
    O, Sf = run(q, k, v, g, zero_b, S0=S0)
    cum = np.exp(np.cumsum(g, axis=0))                     # [T, H, dk]
    Oe = np.einsum("thi,thi,hij->thj", q, cum, S0[0])
    assert rel(O, Oe) < 1e-13, rel(O, Oe)
    assert rel(Sf[0], cum[-1][:, :, None] * S0[0]) < 1e-13


def pin_p3_scalar_gate(run, seed=3):
    rng = np.random.default_rng(seed)
    q, k, v, g, b = rand_inputs(rng, 10, 2, 5, 4)
    g = np.repeat(g[:, :, :1], 5, axis=2)                  # one gate value per (token, head)
    S0 = rng.standard_normal((1, 2, 5, 4))
    O, Sf = run(q, k, v, g, b, S0=S0)
    for h in range(2):
        S = S0[0, h].copy()
        for t in range(10):
            a = np.exp(g[t, h, 0])
            kt = k[t, h][:, None]
            S = a * (np.eye(5) - b[t, h] * kt @ kt.T) @ S + b[t, h] * kt @ v[t, h][None, :]
            assert rel(O[t, h], S.T @ q[t, h]) < 1e-12
        assert rel(Sf[0, h], S) < 1e-12


def pin_p4_exact_write(run, seed=4):
    rng = np.random.default_rng(seed)
    _, _, v, g, _ = rand_inputs(rng, 13, 2, 8, 6)
    # keys exactly unit-norm in fp32: +-1/2 on four random channels
    k = np.zeros((13, 2, 8))
    for t in range(13):
        for h in range(2):
            k[t, h, rng.choice(8, 4, replace=False)] = rng.choice([-0.5, 0.5], 4)
    ones = np.ones((13, 2))
    S0 = rng.standard_normal((1, 2, 8, 6))
    # read with q_t = k_t: o_t = S_t^T k_t, which must be v_t
    O, _ = run(k, k, v, g, ones, S0=S0)
    assert np.max(np.abs(O - v)) < 1e-12, np.max(np.abs(O - v))


def pin_p5_chunk_form(run, seed=5):
    rng = np.random.default_rng(seed)
    q, k, v, g, b = rand_inputs(rng, 37, 2, 8, 6)
    cu = [0, 23, 37]
    S0 = rng.standard_normal((2, 2, 8, 6)) * 0.1
    O, Sf = run(q, k, v, g, b, cu_seqlens=cu, S0=S0)
    for C in (1, 2, 4, 8, 16):
        Oc, Sfc = oracle.chunked.prefill_chunked(q, k, v, g, b, cu, C, S0=S0)
        assert rel(O, Oc) < 1e-11, (C, rel(O, Oc))
        assert rel(Sf, Sfc) < 1e-11, (C, rel(Sf, Sfc))


def pin_p6_lookup_table(run, seed=6):
    rng = np.random.default_rng(seed)
    T, dk, dv = 12, 4, 3
    keys = rng.integers(0, dk, size=T)
    k = np.zeros((T, 1, dk))
    k[np.arange(T), 0, keys] = 1.0
    q = rng.standard_normal((T, 1, dk)).astype(np.float32).astype(np.float64)
    v = rng.standard_normal((T, 1, dv)).astype(np.float32).astype(np.float64)
    O, Sf = run(q, k, v, np.zeros((T, 1, dk)), np.ones((T, 1)))
    table = np.zeros((dk, dv))
    for t in range(T):
        table[keys[t]] = v[t, 0]
        assert np.max(np.abs(O[t, 0] - table.T @ q[t, 0])) < 1e-14
    assert np.max(np.abs(Sf[0, 0] - table)) < 1e-14


def pin_p7_split_and_varlen(run, seed=7):
    rng = np.random.default_rng(seed)
    q, k, v, g, b = rand_inputs(rng, 30, 2, 5, 4)
    S0 = rng.standard_normal((1, 2, 5, 4))
    O, Sf = run(q, k, v, g, b, S0=S0)
    O1, Sf1 = run(q[:13], k[:13], v[:13], g[:13], b[:13], S0=S0)
    O2, Sf2 = run(q[13:], k[13:], v[13:], g[13:], b[13:], S0=Sf1)
    assert rel(np.concatenate([O1, O2]), O) < 1e-13
    assert rel(Sf2, Sf) < 1e-13
    # packed varlen == independent runs
    cu = [0, 7, 7, 19, 30]                                     # includes an empty sequence
    S0v = rng.standard_normal((4, 2, 5, 4))
    Ov, Sfv = run(q, k, v, g, b, cu_seqlens=cu, S0=S0v)
    for n in range(4):
        a, e = cu[n], cu[n + 1]
        On, Sfn = run(q[a:e], k[a:e], v[a:e], g[a:e], b[a:e], S0=S0v[n:n + 1])
        assert rel(Ov[a:e], On) < 1e-15 if e > a else True
        assert np.array_equal(Sfv[n], Sfn[0])
    # ... and without S0 every sequence starts from a zero state, not from the
    # state its predecessor left
    Oz, Sfz = run(q, k, v, g, b, cu_seqlens=cu)
    for n in range(4):
        a, e = cu[n], cu[n + 1]
        On, Sfn = run(q[a:e], k[a:e], v[a:e], g[a:e], b[a:e])
        assert rel(Oz[a:e], On) < 1e-15 if e > a else True
        assert np.array_equal(Sfz[n], Sfn[0])


ALL_PINS = [pin_p1_product_form, pin_p2_no_write, pin_p3_scalar_gate, pin_p4_exact_write,
            pin_p5_chunk_form, pin_p6_lookup_table, pin_p7_split_and_varlen]
