"""The rewrites of the chunk form that the tensor-core path is built on, checked
in fp64 on the CPU against the page's own chunk form (``oracle/chunked.py``)
and the token loop (``oracle.prefill``).

Every identity here is algebra on the "FlashKDA Algorithm" chunk form of the
"Kimi K3: the manos, the mythos, the legendos" page.  The kernels do not
evaluate that form as printed; they evaluate these equivalents:

R1  U = U0 - W S_in with W = INV Diag(beta) K_decay, U0 = INV Diag(beta) V, so
    O = Q' S_in + O0 with Q' = Q_decay - M_qk W and O0 = M_qk U0;
R2  S_out = A_c S_in + B_c, A_c = Diag(a_last) - K_restore^T W,
    B_c = K_restore^T U0; A_c is what a chunk does to S_in = I when V = 0,
    B_c what it does to S_in = 0;
R3  composing those maps over a segment of chunks, scanning the segments'
    maps for their starting states and re-running every segment from its
    starting state gives the token loop's outputs and final state;
R4  (I + L)^-1 from 16x16 diagonal blocks and two levels of 2x2 block merges,
    and in the association the chunk-prep kernel uses (six products of L
    blocks with the diagonal inverses first, so that the chain of dependent
    products is four long);
R5  the Gram weights exp(G_r - G_t) built from per-16-row-block reference
    points stay in the fp32 range at the page's log-decay bound (-5, 0), where
    the page's K_inv = K / a does not.

A slip in any of them (a wrong sign, a transposed factor, a missed
Diag(beta)) fails one of these tests on the CPU, before any GPU run.
"""
from __future__ import annotations

import numpy as np
import pytest
import scipy.linalg

import oracle
from oracle.chunked import chunk_step
from _pins import rand_inputs, rel

C = 64


def chunk_inputs(seed, n=C, dk=128, dv=128, strong_decay=False):
    rng = np.random.default_rng(seed)
    q, k, v, g, beta = rand_inputs(rng, n, 1, dk, dv)
    if strong_decay:
        g = rng.uniform(-5.0, -3.0, size=g.shape).astype(np.float32).astype(np.float64)
    S_in = 0.1 * rng.standard_normal((dk, dv))
    return q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], S_in


def chunk_terms(Q, K, V, g, beta):
    """The state-independent products of one chunk, in the page's notation."""
    n = Q.shape[0]
    a = np.exp(np.cumsum(g, axis=0))
    K_decay, Q_decay, K_inv = a * K, a * Q, K / a
    K_restore = a[-1][None, :] * K_inv
    L = np.tril(beta[:, None] * (K_decay @ K_inv.T), k=-1)
    INV = scipy.linalg.solve_triangular(np.eye(n) + L, np.eye(n), lower=True, unit_diagonal=True)
    M_qk = np.tril(Q_decay @ K_inv.T)
    W = INV @ (beta[:, None] * K_decay)
    U0 = INV @ (beta[:, None] * V)
    return dict(a_last=a[-1], Q_decay=Q_decay, K_restore=K_restore, L=L, INV=INV, M_qk=M_qk, W=W, U0=U0)


@pytest.mark.parametrize("n", [C, 37, 1])
def test_r1_r2_state_independent_forms(n):
    Q, K, V, g, beta, S_in = chunk_inputs(21 + n, n=n)
    O, S_out = chunk_step(Q, K, V, g, beta, S_in)
    t = chunk_terms(Q, K, V, g, beta)
    Q_prime = t["Q_decay"] - t["M_qk"] @ t["W"]
    O0 = t["M_qk"] @ t["U0"]
    assert rel(Q_prime @ S_in + O0, O) < 1e-12
    A_c = np.diag(t["a_last"]) - t["K_restore"].T @ t["W"]
    B_c = t["K_restore"].T @ t["U0"]
    assert rel(A_c @ S_in + B_c, S_out) < 1e-12
    # the two halves of U the state pass forms: U = U0 - W S_in
    U = t["INV"] @ (beta[:, None] * (V - (np.exp(np.cumsum(g, axis=0)) * K) @ S_in))
    assert rel(t["U0"] - t["W"] @ S_in, U) < 1e-12


def test_r1_catches_a_wrong_sign():
    """The check above is not vacuous: Q_decay + M_qk W is far from the truth."""
    Q, K, V, g, beta, S_in = chunk_inputs(5)
    O, _ = chunk_step(Q, K, V, g, beta, S_in)
    t = chunk_terms(Q, K, V, g, beta)
    wrong = (t["Q_decay"] + t["M_qk"] @ t["W"]) @ S_in + t["M_qk"] @ t["U0"]
    assert rel(wrong, O) > 1e-3


def test_r2_map_from_identity_and_zero_runs():
    """A_c and B_c taken the way the first segment pass takes them (a run from
    S_in = I with V = 0, and a run from S_in = 0) reproduce the chunk for any
    starting state."""
    Q, K, V, g, beta, S_in = chunk_inputs(8, dk=64, dv=32)
    dk = K.shape[1]
    _, A_c = chunk_step(Q, K, np.zeros((C, dk)), g, beta, np.eye(dk))
    _, B_c = chunk_step(Q, K, V, g, beta, np.zeros_like(S_in))
    _, S_out = chunk_step(Q, K, V, g, beta, S_in)
    assert rel(A_c @ S_in + B_c, S_out) < 1e-12
    t = chunk_terms(Q, K, V, g, beta)
    assert rel(A_c, np.diag(t["a_last"]) - t["K_restore"].T @ t["W"]) < 1e-12


def segment_scan(q, k, v, g, beta, cu, S0, seg_chunks):
    """Outputs and final states through per-segment affine maps (R3)."""
    T, H, dk = q.shape
    dv = v.shape[2]
    O = np.zeros((T, H, dv))
    Sf = np.zeros((len(cu) - 1, H, dk, dv))
    for n in range(len(cu) - 1):
        bos, eos = int(cu[n]), int(cu[n + 1])
        chunks = [(c0, min(c0 + C, eos)) for c0 in range(bos, eos, C)]
        segments = [chunks[i:i + seg_chunks] for i in range(0, len(chunks), seg_chunks)]
        for h in range(H):
            sl = lambda x, c: x[c[0]:c[1], h]
            # pass 1: every segment as a map from the identity (V = 0) and from zero
            maps = []
            for seg in segments:
                A, B = np.eye(dk), np.zeros((dk, dv))
                for c in seg:
                    _, A = chunk_step(sl(q, c), sl(k, c), np.zeros((c[1] - c[0], dk)), sl(g, c), sl(beta, c), A)
                    _, B = chunk_step(sl(q, c), sl(k, c), sl(v, c), sl(g, c), sl(beta, c), B)
                maps.append((A, B))
            # pass 2: scan over the segments for their starting states
            S = S0[n, h].copy()
            starts = []
            for A, B in maps:
                starts.append(S)
                S = A @ S + B
            Sf[n, h] = S
            # pass 3: every segment from its starting state, writing O
            for seg, S in zip(segments, starts):
                for c in seg:
                    O[c[0]:c[1], h], S = chunk_step(sl(q, c), sl(k, c), sl(v, c), sl(g, c), sl(beta, c), S)
    return O, Sf


@pytest.mark.parametrize("seg_chunks", [1, 3, 16])
def test_r3_segment_scan_equals_token_loop(seg_chunks):
    rng = np.random.default_rng(30 + seg_chunks)
    lengths = [C * 13 + 29, 0, 100, C * 2]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    T, H, dk, dv = int(cu[-1]), 2, 32, 16
    q, k, v, g, beta = rand_inputs(rng, T, H, dk, dv)
    S0 = 0.1 * rng.standard_normal((len(lengths), H, dk, dv))
    O, Sf = segment_scan(q, k, v, g, beta, cu, S0, seg_chunks)
    O_ref, Sf_ref = oracle.prefill(q, k, v, g, beta, cu_seqlens=cu, S0=S0)
    assert rel(O, O_ref) < 1e-10
    assert rel(Sf, Sf_ref) < 1e-10


def block_merge_inverse(L, b=16):
    """(I + L)^-1 for strictly lower L: b x b diagonal blocks by forward
    substitution, then merges [[A, 0], [X, D]]^-1 = [[A^-1, 0], [-D^-1 X A^-1, D^-1]]
    of neighbouring blocks until one block covers the matrix."""
    n = L.shape[0]
    M = np.eye(n) + L
    INV = np.zeros_like(M)
    for s in range(0, n, b):
        e = min(s + b, n)
        for i in range(s, e):                     # row i of the block's inverse
            INV[i, i] = 1.0
            for j in range(s, i):
                INV[i, j] = -sum(M[i, m] * INV[m, j] for m in range(j, i))
    w = b
    while w < n:
        for s in range(0, n, 2 * w):
            m, e = min(s + w, n), min(s + 2 * w, n)
            if m >= e:
                continue
            INV[m:e, s:m] = -INV[m:e, m:e] @ M[m:e, s:m] @ INV[s:m, s:m]
        w *= 2
    return INV


@pytest.mark.parametrize("n", [C, 50, 16])
def test_r4_block_merge_inverse(n):
    Q, K, V, g, beta, _ = chunk_inputs(40 + n, n=n, dk=32, dv=8)
    L = chunk_terms(Q, K, V, g, beta)["L"]
    ref = scipy.linalg.solve_triangular(np.eye(n) + L, np.eye(n), lower=True, unit_diagonal=True)
    assert rel(block_merge_inverse(L), ref) < 1e-12
    assert np.max(np.abs(block_merge_inverse(L) @ (np.eye(n) + L) - np.eye(n))) < 1e-12


def four_block_inverse(L, b=16):
    """(I + L)^-1 for a 4b x 4b strictly lower L the way the chunk-prep kernel
    associates it: diagonal inverses D_i, then six products that need only
    them, F = L10 D0, E = L32 D2, B0 = L21 D1, B1 = L31 D1, C0 = L20 D0,
    C1 = L30 D0; then INV_10 = -D1 F, INV_32 = -D3 E and the blocks of
    Z = L_[23][01] INV_top as Z00 = C0 - B0 F, Z10 = C1 - B1 F, Z01 = B0,
    Z11 = B1; finally the lower-left quarter -INV_bottom Z."""
    M = np.eye(4 * b) + L
    blk = lambda X, i, j: X[b * i:b * (i + 1), b * j:b * (j + 1)]
    D = [np.linalg.inv(blk(M, i, i)) for i in range(4)]
    F, E = blk(L, 1, 0) @ D[0], blk(L, 3, 2) @ D[2]
    B0, B1 = blk(L, 2, 1) @ D[1], blk(L, 3, 1) @ D[1]
    C0, C1 = blk(L, 2, 0) @ D[0], blk(L, 3, 0) @ D[0]
    I10, I32 = -D[1] @ F, -D[3] @ E
    Z00, Z10 = C0 - B0 @ F, C1 - B1 @ F
    INV = np.zeros_like(M)
    for i in range(4):
        INV[b * i:b * (i + 1), b * i:b * (i + 1)] = D[i]
    INV[b:2 * b, 0:b], INV[3 * b:4 * b, 2 * b:3 * b] = I10, I32
    INV[2 * b:3 * b, 0:b] = -D[2] @ Z00
    INV[2 * b:3 * b, b:2 * b] = -D[2] @ B0
    INV[3 * b:4 * b, 0:b] = -(I32 @ Z00 + D[3] @ Z10)
    INV[3 * b:4 * b, b:2 * b] = -(I32 @ B0 + D[3] @ B1)
    return INV


@pytest.mark.parametrize("strong_decay", [False, True])
def test_r4_four_block_association_of_the_kernel(strong_decay):
    """The 64 x 64 inverse in the kernel's association equals the triangular
    solve, at both ends of the decay range."""
    Q, K, V, g, beta, _ = chunk_inputs(60 + strong_decay, dk=32, dv=8, strong_decay=strong_decay)
    L = chunk_terms(Q, K, V, g, beta)["L"]
    ref = scipy.linalg.solve_triangular(np.eye(C) + L, np.eye(C), lower=True, unit_diagonal=True)
    assert rel(four_block_inverse(L), ref) < 1e-12
    assert np.max(np.abs(four_block_inverse(L) @ (np.eye(C) + L) - np.eye(C))) < 1e-12


def test_r5_block_reference_staging_stays_in_fp32_range():
    """At the bound log alpha -> -5 the cumulative log-decay of a 64-token chunk
    reaches -320: exp(+320) overflows fp32, so the page's K_inv = K / a cannot
    be formed there.  Per 16-row block b with reference row p_b = 16 b, the row
    factors exp(G_r - G_pb) (r in the block) and column factors
    exp(G_pb - G_t) (t < p_b + 16) stay finite in fp32, and their products give
    the exact weights of M_qk = tril(Q_decay K_inv^T) and L."""
    Q, K, V, g, beta, _ = chunk_inputs(50, strong_decay=True)
    g32 = g.astype(np.float32)
    G = np.cumsum(g32, axis=0, dtype=np.float32)           # fp32, as on the GPU
    with np.errstate(over="ignore"):
        assert not np.all(np.isfinite(np.exp(-G)))         # the page's K_inv = K / a overflows
    Gd = G.astype(np.float64)
    # exact weights from the same fp32 cumulative sums, in fp64
    Wexact = np.exp(Gd[:, None, :] - Gd[None, :, :])       # [r, t, channel]
    r_idx = np.arange(C)[:, None, None]
    t_idx = np.arange(C)[None, :, None]
    M_exact = np.einsum("rj,tj,rtj->rt", Q, K, np.where(r_idx >= t_idx, Wexact, 0.0))
    L_exact = beta[:, None] * np.einsum("rj,tj,rtj->rt", K, K, np.where(r_idx > t_idx, Wexact, 0.0))
    M = np.zeros((C, C))
    L = np.zeros((C, C))
    for b in range(C // 16):
        p = 16 * b
        rows, cols = slice(p, p + 16), slice(0, p + 16)
        e_row = G[rows] - G[p]
        e_col = G[p] - G[cols]
        assert e_row.max() <= 0 and e_row.min() >= -75                 # row factors <= 1
        assert e_col[p:].min() >= 0 and e_col[p:].max() <= 75          # own block: <= e^75
        if p:
            assert e_col[:p].max() <= 0                                # earlier rows: <= 1
        rf = np.exp(e_row.astype(np.float32))
        cf = np.exp(e_col.astype(np.float32))
        assert np.all(np.isfinite(rf)) and np.all(np.isfinite(cf))
        Mq = (Q[rows] * rf) @ (K[cols] * cf).T
        Mk = (K[rows] * rf) @ (K[cols] * cf).T
        r = np.arange(p, p + 16)[:, None]
        t = np.arange(0, p + 16)[None, :]
        M[rows, cols] = np.where(t <= r, Mq, 0.0)
        L[rows, cols] = np.where(t < r, beta[rows][:, None] * Mk, 0.0)
    scale_m = np.max(np.abs(M_exact))
    assert np.max(np.abs(M - M_exact)) <= 1e-5 * scale_m
    assert np.max(np.abs(L - L_exact)) <= 1e-5 * np.max(np.abs(L_exact))
