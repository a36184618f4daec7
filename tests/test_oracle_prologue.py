"""Pins of the oracle's fused prologue (CPU only).

The prologue is the parameter-free front of the Kimi Linear layer: q and k
L2-normalised ("Kimi K3: the manos, the mythos, the legendos", section "Kimi
Linear"), log-decay = clamp(-softplus(gate), -5, -1e-4) (the (-5, 0) bound of
"LLM architecture at trillion scale", section "The KDA update, in plain
words") and beta = sigmoid(beta_logit).  Each check below uses an identity
other than the oracle's own formula."""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def test_unit_rows_are_unit_and_parallel():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((40, 128)) * rng.uniform(0.1, 20.0, (40, 1))).astype(np.float32)
    xh, _, _ = oracle.prologue(x=x)
    xd = x.astype(np.float64)
    ss = (xd * xd).sum(axis=1)
    # |x_hat|^2 = |x|^2 / (|x|^2 + eps)
    assert np.allclose((xh * xh).sum(axis=1), ss / (ss + 1e-6), rtol=0, atol=1e-13)
    # Cauchy-Schwarz with equality: x_hat is a positive multiple of x
    dot = (xh * xd).sum(axis=1)
    assert np.all(dot > 0)
    assert np.allclose(dot * dot, (xh * xh).sum(axis=1) * ss, rtol=1e-12, atol=0)


def test_zero_row_stays_zero():
    xh, _, _ = oracle.prologue(x=np.zeros((2, 32), dtype=np.float32))
    assert np.all(xh == 0.0)


def test_log_decay_is_log_of_sigmoid_and_clamped():
    a = np.linspace(-30.0, 30.0, 2001).astype(np.float32)
    _, la, _ = oracle.prologue(gate=a)
    ad = a.astype(np.float64)
    # -softplus(a) = log(sigmoid(-a)) = log(1 / (1 + e^a)), clamped to [-5, -1e-4]
    ref = np.clip(np.log(1.0 / (1.0 + np.exp(ad))), -5.0, -1e-4)
    assert np.allclose(la, ref, rtol=1e-12, atol=1e-15)
    assert la.min() == -5.0 and la.max() == -1e-4
    _, l0, _ = oracle.prologue(gate=np.zeros(1, dtype=np.float32))
    assert abs(l0[0] + np.log(2.0)) < 1e-15


def test_beta_is_a_logistic():
    b = np.linspace(-12.0, 12.0, 97).astype(np.float32)
    _, _, bp = oracle.prologue(beta_logit=b)
    _, _, bm = oracle.prologue(beta_logit=-b)
    assert np.allclose(bp + bm, 1.0, rtol=0, atol=1e-15)                     # symmetry
    assert np.allclose(np.log(bp / (1.0 - bp)), b.astype(np.float64), atol=1e-9)   # logit inverts it
    assert np.all((bp > 0) & (bp < 1))


def test_fused_prefill_routes_the_prologue_outputs():
    """Raw inputs built so that the prologue returns chosen values (scaled unit
    rows; gate = inverse softplus of -log_alpha; beta_logit = logit(beta)):
    the fused oracle must then equal the plain oracle on those values."""
    rng = np.random.default_rng(7)
    T, H, dk, dv = 37, 2, 16, 8
    qu = rng.standard_normal((T, H, dk)); qu /= np.linalg.norm(qu, axis=-1, keepdims=True)
    ku = rng.standard_normal((T, H, dk)); ku /= np.linalg.norm(ku, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv)).astype(np.float32)
    g = rng.uniform(-4.0, -0.01, (T, H, dk))
    beta = rng.uniform(0.05, 0.95, (T, H))
    gate = np.log(np.expm1(-g)).astype(np.float32)            # -softplus(gate) = g
    beta_logit = np.log(beta / (1.0 - beta)).astype(np.float32)
    s_q, s_k = 3.5, 0.25
    q_raw = (qu * s_q).astype(np.float32)
    k_raw = (ku * s_k).astype(np.float32)
    cu = [0, 20, T]
    S0 = rng.standard_normal((2, H, dk, dv)) * 0.1
    # what the prologue yields, from the same fp32 raw values
    q_in = q_raw.astype(np.float64) / np.sqrt((q_raw.astype(np.float64) ** 2).sum(-1, keepdims=True) + 1e-6)
    k_in = k_raw.astype(np.float64) / np.sqrt((k_raw.astype(np.float64) ** 2).sum(-1, keepdims=True) + 1e-6)
    O_f, S_f = oracle.prefill_fused(q_raw, k_raw, v, gate, beta_logit, cu_seqlens=cu, S0=S0)
    O_p, S_p = oracle.prefill(q_in.astype(np.float32), k_in.astype(np.float32), v, g.astype(np.float32),
                              beta.astype(np.float32), cu_seqlens=cu, S0=S0)
    assert np.max(np.abs(O_f - O_p)) / np.max(np.abs(O_p)) < 1e-5
    assert np.max(np.abs(S_f - S_p)) / np.max(np.abs(S_p)) < 1e-5
    # and a swapped routing (q and k exchanged) is far off
    O_x, _ = oracle.prefill_fused(k_raw, q_raw, v, gate, beta_logit, cu_seqlens=cu, S0=S0)
    assert np.max(np.abs(O_x - O_p)) / np.max(np.abs(O_p)) > 1e-2
