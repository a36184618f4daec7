"""Seeded synthetic inputs for KDA prefill and decode.

This module is shared by the tests, the benchmark and the smoke check, and
feeds both the CUDA path and the CPU oracle.  It holds none of the method's
arithmetic: it only draws random tensors and shapes them like the pages'
workloads.  The per-tensor recipe is

* q, k ~ N(0, 1), L2-normalised over d_k per (token, head) in fp32, then cast to
  the storage dtype (the Kimi Linear layer normalises q and k before the
  operator -- "Kimi K3: the manos, the mythos, the legendos", section
  "Kimi Linear");
* v ~ N(0, 1) in the storage dtype;
* beta = sigmoid(N(0, 1)), fp32, one per (token, head);
* log_alpha = clamp(-softplus(N(mu, 1)), -5, -1e-4), fp32, one per
  (token, head, key channel) -- the log-decay bound (-5, 0) of the
  "LLM architecture at trillion scale" page, section "The KDA update, in plain
  words";
* S0 ~ N(0, 0.02^2) fp32 where a workload asks for a non-zero initial state.

Draw order on one ``torch.Generator``: q, k, v, beta-logits, gate-logits, S0.
Variable lengths are drawn first from ``numpy.random.default_rng(seed)``.

``raw=True`` returns the same draws before the normalisation and the two
activations (q, k ~ N(0, 1) cast to the storage dtype; gate = N(mu, 1) and
beta_logit = N(0, 1) in fp32), the inputs of the fused-prologue entry points.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    kind: str               # "prefill" or "decode"
    H: int
    dk: int
    dv: int
    dtype: torch.dtype      # storage dtype of q, k, v and O
    chunk: int = 64
    T: int = 0              # tokens per sequence (fixed-length prefill)
    B: int = 1              # sequences (fixed-length prefill) / decode batch N
    varlen: tuple = ()      # (n_seq, lo, hi): lengths uniform in [lo, hi]
    gate_mu: float = 0.0
    s0_std: float = 0.0     # 0 -> S0 = None (zeros)
    steps: int = 1          # decode: consecutive in-place steps


WORKLOADS = {
    # tiny fp32 correctness case
    "tiny_fp32_T64_H2_D32": Workload("tiny_fp32_T64_H2_D32", "prefill", H=2, dk=32, dv=32,
                                     dtype=torch.float32, chunk=16, T=64, B=1),
    # single 8K-token sequence, 32 heads of 128
    "prefill_bf16_T8192_H32_D128": Workload("prefill_bf16_T8192_H32_D128", "prefill", H=32, dk=128,
                                            dv=128, dtype=torch.bfloat16, chunk=64, T=8192, B=1),
    # 8 packed sequences of 1K..32K tokens with random initial states
    "varlen_bf16_8seq_1K_32K_H32_D128": Workload("varlen_bf16_8seq_1K_32K_H32_D128", "prefill", H=32,
                                                 dk=128, dv=128, dtype=torch.bfloat16, chunk=64,
                                                 varlen=(8, 1024, 32768), s0_std=0.02),
    # 256 sequences x 32 heads, one token each, 1000 in-place steps
    "decode_bf16_N256_H32_D128": Workload("decode_bf16_N256_H32_D128", "decode", H=32, dk=128, dv=128,
                                          dtype=torch.bfloat16, B=256, s0_std=0.02, steps=1000),
    # one 1,048,576-token sequence with strong-decay gates
    "long_bf16_T1M_H32_D128": Workload("long_bf16_T1M_H32_D128", "prefill", H=32, dk=128, dv=128,
                                       dtype=torch.bfloat16, chunk=64, T=1 << 20, B=1, gate_mu=1.0),
}


def seq_lengths(w: Workload, seed: int = 0):
    """Per-sequence lengths (host list)."""
    if w.varlen:
        n, lo, hi = w.varlen
        return [int(x) for x in np.random.default_rng(seed).integers(lo, hi + 1, size=n)]
    return [w.T] * w.B


def _normal(shape, gen, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)


def _unit_rows(x):
    return x / torch.linalg.vector_norm(x, dim=-1, keepdim=True).clamp_min(1e-12)


def make_qkv_gates(T, H, dk, dv, dtype, gen, device, gate_mu=0.0, raw=False):
    """q, k, v, beta, log_alpha for T packed tokens, in the draw order above
    (raw: q, k, v, beta_logit, gate before the normalisation and activations)."""
    q = _normal((T, H, dk), gen, device)
    k = _normal((T, H, dk), gen, device)
    v = _normal((T, H, dv), gen, device).to(dtype)
    b = _normal((T, H), gen, device)
    a = _normal((T, H, dk), gen, device) + gate_mu
    if raw:
        return q.to(dtype).contiguous(), k.to(dtype).contiguous(), v.contiguous(), b.contiguous(), a.contiguous()
    q = _unit_rows(q).to(dtype)
    k = _unit_rows(k).to(dtype)
    beta = torch.sigmoid(b)
    log_alpha = (-torch.nn.functional.softplus(a)).clamp(-5.0, -1e-4)
    return q.contiguous(), k.contiguous(), v.contiguous(), beta.contiguous(), log_alpha.contiguous()


def make_prefill(w: Workload, device="cpu", seed: int = 0, lengths=None, raw=False):
    """Inputs for a prefill workload: dict with q, k, v, log_alpha, beta, S0,
    cu_seqlens (int32, on ``device``), cu_seqlens_host (list) and lengths.
    raw=True: gate and beta_logit in place of log_alpha and beta, q and k not
    normalised."""
    lens = list(lengths) if lengths is not None else seq_lengths(w, seed)
    T = int(sum(lens))
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    q, k, v, beta, log_alpha = make_qkv_gates(T, w.H, w.dk, w.dv, w.dtype, gen, device, w.gate_mu, raw)
    S0 = None
    if w.s0_std > 0:
        S0 = (_normal((len(lens), w.H, w.dk, w.dv), gen, device) * w.s0_std).contiguous()
    cu_host = [0]
    for L in lens:
        cu_host.append(cu_host[-1] + L)
    cu = torch.tensor(cu_host, dtype=torch.int32, device=device)
    gates = dict(gate=log_alpha, beta_logit=beta) if raw else dict(log_alpha=log_alpha, beta=beta)
    return dict(q=q, k=k, v=v, S0=S0, cu_seqlens=cu, cu_seqlens_host=cu_host, lengths=lens, T=T, **gates)


def make_decode(w: Workload, device="cpu", seed: int = 0, n_token_sets: int = 1, raw=False):
    """State plus ``n_token_sets`` fresh one-token sets for a decode workload.

    Returns dict with S [N, H, dk, dv] fp32 and lists q, k, v, log_alpha, beta
    (one [N, H, .] tensor per set); raw=True: gate, beta_logit instead."""
    N = w.B
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    sets = [make_qkv_gates(N, w.H, w.dk, w.dv, w.dtype, gen, device, w.gate_mu, raw)
            for _ in range(n_token_sets)]
    S = (_normal((N, w.H, w.dk, w.dv), gen, device) * (w.s0_std if w.s0_std > 0 else 0.02)).contiguous()
    q, k, v, beta, log_alpha = (list(x) for x in zip(*sets))
    if raw:
        return dict(q=q, k=k, v=v, beta_logit=beta, gate=log_alpha, S=S)
    return dict(q=q, k=k, v=v, beta=beta, log_alpha=log_alpha, S=S)
