"""The seeded input generator follows its stated recipe (CPU only): workload
sizes, value distributions, the log-decay clamp, seed determinism, and the
raw draws of the fused-prologue entry points being the same random numbers."""
import numpy as np
import pytest
import torch

from kimi_delta_attention_chunked_gb300 import inputs


def expect(f, mu=0.0):
    """E[f(Z)] for Z ~ N(mu, 1), by quadrature."""
    z = np.linspace(mu - 12.0, mu + 12.0, 200001)
    w = np.exp(-0.5 * (z - mu) ** 2) / np.sqrt(2 * np.pi)
    return float(np.trapezoid(f(z) * w, z))


def test_workload_sizes():
    W = inputs.WORKLOADS
    t = W["tiny_fp32_T64_H2_D32"]
    assert (t.H, t.dk, t.dv, t.T, t.B, t.chunk, t.dtype, t.s0_std) == (2, 32, 32, 64, 1, 16, torch.float32, 0.0)
    p = W["prefill_bf16_T8192_H32_D128"]
    assert (p.H, p.dk, p.dv, p.T, p.B, p.chunk, p.dtype, p.s0_std) == (32, 128, 128, 8192, 1, 64, torch.bfloat16, 0.0)
    v = W["varlen_bf16_8seq_1K_32K_H32_D128"]
    assert v.varlen == (8, 1024, 32768) and (v.H, v.dk, v.s0_std, v.dtype) == (32, 128, 0.02, torch.bfloat16)
    d = W["decode_bf16_N256_H32_D128"]
    assert (d.B, d.H, d.dk, d.dv, d.s0_std, d.steps, d.dtype) == (256, 32, 128, 128, 0.02, 1000, torch.bfloat16)
    g = W["long_bf16_T1M_H32_D128"]
    assert (g.T, g.H, g.dk, g.gate_mu, g.dtype) == (1 << 20, 32, 128, 1.0, torch.bfloat16)


def test_varlen_lengths_are_seeded_and_in_range():
    w = inputs.WORKLOADS["varlen_bf16_8seq_1K_32K_H32_D128"]
    a, b = inputs.seq_lengths(w, 0), inputs.seq_lengths(w, 0)
    assert a == b and len(a) == 8 and all(1024 <= x <= 32768 for x in a)
    assert inputs.seq_lengths(w, 1) != a


@pytest.mark.parametrize("mu", [0.0, 1.0])
def test_prefill_distributions(mu):
    w = inputs.Workload("dist", "prefill", H=4, dk=128, dv=64, dtype=torch.bfloat16, T=2048, B=1, gate_mu=mu,
                        s0_std=0.02)
    d = inputs.make_prefill(w, seed=3)
    T, H = 2048, 4
    assert d["q"].shape == (T, H, 128) and d["v"].shape == (T, H, 64) and d["beta"].shape == (T, H)
    assert d["q"].dtype == torch.bfloat16 and d["log_alpha"].dtype == torch.float32
    assert d["S0"].shape == (1, H, 128, 64)
    # q and k: unit rows before the bf16 cast (bf16 keeps the norm within a few 1e-3)
    for x in (d["q"], d["k"]):
        n = torch.linalg.vector_norm(x.float(), dim=-1)
        assert torch.all((n - 1).abs() < 1e-2)
    # v ~ N(0, 1)
    vv = d["v"].float()
    assert abs(vv.mean().item()) < 0.02 and abs(vv.std().item() - 1) < 0.02
    # beta = sigmoid(N(0, 1))
    b = d["beta"].double().numpy()
    assert np.all((b > 0) & (b < 1))
    assert abs(b.mean() - expect(lambda z: 1 / (1 + np.exp(-z)))) < 0.01
    # log_alpha = clamp(-softplus(N(mu, 1)), -5, -1e-4)
    g = d["log_alpha"].double().numpy()
    assert g.min() >= -5.0 and g.max() <= -1e-4 + 1e-9
    ref = expect(lambda z: np.clip(-np.log1p(np.exp(z)), -5.0, -1e-4), mu)
    assert abs(g.mean() - ref) < 0.01, (g.mean(), ref)
    # S0 ~ N(0, 0.02^2)
    assert abs(d["S0"].std().item() - 0.02) < 0.001


def test_seeded_and_reproducible():
    w = inputs.WORKLOADS["tiny_fp32_T64_H2_D32"]
    a, b, c = inputs.make_prefill(w, seed=5), inputs.make_prefill(w, seed=5), inputs.make_prefill(w, seed=6)
    for key in ("q", "k", "v", "log_alpha", "beta"):
        assert torch.equal(a[key], b[key])
        assert not torch.equal(a[key], c[key])


def test_raw_draws_are_the_same_random_numbers():
    """raw=True returns the draws before normalisation and activations: applying
    them gives back the normal draws of the same seed exactly."""
    w = inputs.Workload("raw", "prefill", H=2, dk=32, dv=16, dtype=torch.float32, T=100, B=1, gate_mu=0.5)
    d = inputs.make_prefill(w, seed=9)
    r = inputs.make_prefill(w, seed=9, raw=True)
    unit = lambda x: x / torch.linalg.vector_norm(x, dim=-1, keepdim=True).clamp_min(1e-12)
    assert torch.equal(unit(r["q"]), d["q"]) and torch.equal(unit(r["k"]), d["k"])
    assert torch.equal(r["v"], d["v"])
    assert torch.equal(torch.sigmoid(r["beta_logit"]), d["beta"])
    assert torch.equal((-torch.nn.functional.softplus(r["gate"])).clamp(-5.0, -1e-4), d["log_alpha"])


def test_decode_token_sets():
    w = inputs.Workload("dec", "decode", H=3, dk=64, dv=32, dtype=torch.bfloat16, B=5, s0_std=0.02)
    d = inputs.make_decode(w, seed=2, n_token_sets=4)
    assert len(d["q"]) == 4 and d["q"][0].shape == (5, 3, 64) and d["v"][0].shape == (5, 3, 32)
    assert d["S"].shape == (5, 3, 64, 32) and d["S"].dtype == torch.float32
    assert not torch.equal(d["q"][0], d["q"][1])                    # a fresh token set per step
