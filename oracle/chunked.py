"""FlashKDA chunk form of KDA, in fp64 numpy -- a cross-check of the oracle.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

This restates, step by step and in the pages' own order and notation, the
chunked matrix form that the "Kimi K3: the manos, the mythos, the legendos"
page (section "FlashKDA Algorithm", sub-section "Algorithm") derives from the
per-token recurrence.  For a chunk of tokens with starting state S_in:

    a          = exp(cumsum(g))                  (inclusive, per key channel)
    K_decay    = Diag(a) K,  Q_decay = Diag(a) Q
    K_inv      = Diag(a)^-1 K
    K_restore  = a[-1] * K_inv
    L          = StrictTril(Diag(beta) K_decay K_inv^T)
    INV        = (I + L)^-1
    M_qk       = tril(Q_decay K_inv^T)
    U          = INV Diag(beta) (V - K_decay S_in)
    O          = Q_decay S_in + M_qk U
    S_out      = Diag(a[-1]) S_in + K_restore^T U

(The page writes exp2 for FlashKDA's internal base-2 gate; here g is the
natural log of alpha, so exp is used.)  In fp64, K_inv stays finite for the
small chunks this is used with (|cumsum g| <= 5 C), so no staging is needed.
The triangular inverse is a library solve, which is a step the form names.

Nothing here is used by the CUDA path.  Its job is pin P5: this form and the
token loop in ``kda_ref.c`` must agree to rounding for every chunk size.
"""
from __future__ import annotations

import numpy as np
import scipy.linalg


def chunk_step(Q, K, V, g, beta, S_in):
    """One chunk.  Q, K, g: [n, dk]; V: [n, dv]; beta: [n]; S_in: [dk, dv].

    Returns (O [n, dv], S_out [dk, dv]).  All fp64.
    """
    n = Q.shape[0]
    a = np.exp(np.cumsum(g, axis=0))            # [n, dk], inclusive cumulative decay
    K_decay = a * K
    Q_decay = a * Q
    K_inv = K / a
    K_restore = a[-1][None, :] * K_inv
    L = np.tril(beta[:, None] * (K_decay @ K_inv.T), k=-1)
    I = np.eye(n)
    INV = scipy.linalg.solve_triangular(I + L, I, lower=True, unit_diagonal=True)
    M_qk = np.tril(Q_decay @ K_inv.T)
    U = INV @ (beta[:, None] * (V - K_decay @ S_in))
    O = Q_decay @ S_in + M_qk @ U
    S_out = a[-1][:, None] * S_in + K_restore.T @ U
    return O, S_out


def prefill_chunked(q, k, v, log_alpha, beta, cu_seqlens, chunk, S0=None):
    """Packed varlen prefill in the chunk form.

    q, k, log_alpha: [T, H, dk]; v: [T, H, dv]; beta: [T, H]; cu_seqlens: [n_seq+1];
    S0: [n_seq, H, dk, dv] or None.  Chunks restart at every sequence start and
    the last chunk of a sequence may be short.  Returns (O [T, H, dv],
    S_final [n_seq, H, dk, dv]) in fp64.
    """
    q, k, v, log_alpha, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, log_alpha, beta))
    T, H, dk = q.shape
    dv = v.shape[2]
    n_seq = len(cu_seqlens) - 1
    O = np.zeros((T, H, dv))
    S_final = np.zeros((n_seq, H, dk, dv))
    for n in range(n_seq):
        bos, eos = int(cu_seqlens[n]), int(cu_seqlens[n + 1])
        for h in range(H):
            S = np.zeros((dk, dv)) if S0 is None else np.array(S0[n, h], dtype=np.float64)
            for c0 in range(bos, eos, chunk):
                c1 = min(c0 + chunk, eos)
                O[c0:c1, h], S = chunk_step(q[c0:c1, h], k[c0:c1, h], v[c0:c1, h],
                                            log_alpha[c0:c1, h], beta[c0:c1, h], S)
            S_final[n, h] = S
    return O, S_final
