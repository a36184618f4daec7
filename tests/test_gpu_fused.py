"""Fused-prologue entry points (q, k normalisation and the gate / beta
activations inside the kernels) vs the fp64 oracle with the same prologue."""
import pytest
import torch

import oracle
import kimi_delta_attention_chunked_gb300 as kda
from kimi_delta_attention_chunked_gb300 import inputs
from _gpu import need_gpu, rel_err, tol_for

pytestmark = pytest.mark.gpu


def run_fused(w, dev, lengths, seed=0, heads=None):
    d = inputs.make_prefill(w, device=dev, seed=seed, lengths=lengths, raw=True)
    O, Sf = kda.kda_prefill_fused(d["q"], d["k"], d["v"], d["gate"], d["beta_logit"], S0=d["S0"],
                                  cu_seqlens=d["cu_seqlens"], cu_seqlens_host=d["cu_seqlens_host"],
                                  chunk=w.chunk)
    torch.cuda.synchronize()
    assert kda.kda_get_last_device_status() == 0
    h0, h1 = heads or (0, w.H)
    sl = slice(h0, h1)
    c = lambda t: t[:, sl].contiguous()
    O_ref, S_ref = oracle.prefill_fused(c(d["q"]), c(d["k"]), c(d["v"]), c(d["gate"]), c(d["beta_logit"]),
                                        cu_seqlens=d["cu_seqlens_host"],
                                        S0=None if d["S0"] is None else d["S0"][:, sl].contiguous())
    eo, es = rel_err(O[:, sl], O_ref), rel_err(Sf[:, sl], S_ref)
    print(f"PARITY fused {w.name} dtype={w.dtype} lengths={d['lengths'][:4]} heads={h0}:{h1} "
          f"O={eo:.3e} S={es:.3e}")
    return eo, es


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dk,dv,chunk", [(32, 32, 16), (64, 128, 32), (128, 64, 64)])
def test_fused_simt(dtype, dk, dv, chunk):
    dev = need_gpu()
    w = inputs.Workload("fused_simt", "prefill", H=3, dk=dk, dv=dv, dtype=dtype, chunk=chunk, s0_std=0.02)
    eo, es = run_fused(w, dev, [0, 1, chunk - 1, 2 * chunk + 7], seed=dk + dv)
    assert eo <= tol_for(dtype) and es <= tol_for(dtype), (eo, es)


def test_fused_tiny_fp32():
    dev = need_gpu()
    w = inputs.WORKLOADS["tiny_fp32_T64_H2_D32"]
    eo, es = run_fused(w, dev, None)
    assert eo <= 1e-4 and es <= 1e-4, (eo, es)


def test_fused_tensor_core_varlen():
    dev = need_gpu()
    w = inputs.Workload("fused_tc", "prefill", H=4, dk=128, dv=128, dtype=torch.bfloat16, chunk=64, s0_std=0.02)
    eo, es = run_fused(w, dev, [0, 130, 1, 640, 63, 257], seed=4)
    assert eo <= tol_for(w.dtype) and es <= tol_for(w.dtype), (eo, es)


def test_fused_full_size_prefill():
    """B = 1, T = 8192, H = 32, d = 128 from raw logits; heads sampled for the oracle."""
    dev = need_gpu()
    w = inputs.WORKLOADS["prefill_bf16_T8192_H32_D128"]
    eo, es = run_fused(w, dev, None, heads=(5, 7))
    assert eo <= tol_for(w.dtype) and es <= tol_for(w.dtype), (eo, es)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dk,dv", [(32, 64), (128, 128)])
def test_fused_decode(dtype, dk, dv):
    dev = need_gpu()
    w = inputs.Workload("fused_dec", "decode", H=4, dk=dk, dv=dv, dtype=dtype, B=16, s0_std=0.02)
    d = inputs.make_decode(w, device=dev, seed=dk, raw=True)
    S = d["S"].clone()
    o = kda.kda_decode_fused(d["q"][0], d["k"][0], d["v"][0], d["gate"][0], d["beta_logit"][0], S)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.decode_fused(d["q"][0], d["k"][0], d["v"][0], d["gate"][0], d["beta_logit"][0],
                                       d["S"].cpu())
    eo, es = rel_err(o, o_ref), rel_err(S, S_ref)
    print(f"PARITY fused decode dtype={dtype} dk={dk} dv={dv} o={eo:.3e} S={es:.3e}")
    assert eo <= tol_for(dtype) and es <= tol_for(dtype), (eo, es)


def test_fused_tensor_core_no_decay():
    """The fused tensor-core prep at the no-decay end: gate pre-activations of
    -40 give log alpha at the upper clamp (-1e-4) on every channel, and beta
    logits of +20 give beta ~ 1, so the prep takes its f16 Gram operands in
    the prologue instantiation too."""
    dev = need_gpu()
    w = inputs.Workload("fused_nodecay", "prefill", H=4, dk=128, dv=128, dtype=torch.bfloat16, chunk=64,
                        s0_std=0.02)
    d = inputs.make_prefill(w, device=dev, seed=23, lengths=[2048 + 29], raw=True)
    d["gate"].fill_(-40.0)
    d["beta_logit"].fill_(20.0)
    O, Sf = kda.kda_prefill_fused(d["q"], d["k"], d["v"], d["gate"], d["beta_logit"], S0=d["S0"],
                                  cu_seqlens=d["cu_seqlens"], cu_seqlens_host=d["cu_seqlens_host"], chunk=64)
    torch.cuda.synchronize()
    assert kda.kda_get_last_device_status() == 0
    O_ref, S_ref = oracle.prefill_fused(d["q"], d["k"], d["v"], d["gate"], d["beta_logit"],
                                        cu_seqlens=d["cu_seqlens_host"], S0=d["S0"])
    eo, es = rel_err(O, O_ref), rel_err(Sf, S_ref)
    print(f"PARITY fused no-decay tc O={eo:.3e} S={es:.3e}")
    assert eo <= 5e-3 and es <= 5e-3, (eo, es)
