"""Decode step: CUDA kernel vs the fp64 oracle (one token per sequence)."""
import numpy as np
import pytest
import torch

import oracle
import kimi_delta_attention_chunked_gb300 as kda
from kimi_delta_attention_chunked_gb300 import inputs
from _gpu import need_gpu, rel_err, tol_for

pytestmark = pytest.mark.gpu


def _run_steps(w, steps, dev, seed=0):
    d = inputs.make_decode(w, device=dev, seed=seed, n_token_sets=steps)
    S = d["S"].clone()
    S_ref = d["S"].double().cpu().numpy()
    worst_o = worst_s = 0.0
    for t in range(steps):
        o = kda.kda_decode(d["q"][t], d["k"][t], d["v"][t], d["log_alpha"][t], d["beta"][t], S)
        o_ref, S_ref = oracle.decode(d["q"][t], d["k"][t], d["v"][t], d["log_alpha"][t], d["beta"][t], S_ref)
        worst_o = max(worst_o, rel_err(o, o_ref))
        worst_s = max(worst_s, rel_err(S, S_ref))
    assert kda.kda_get_last_device_status() == 0
    return worst_o, worst_s


def test_decode_full_size_bf16():
    """256 sequences x 32 heads x d=128, three consecutive in-place steps."""
    dev = need_gpu()
    w = inputs.WORKLOADS["decode_bf16_N256_H32_D128"]
    eo, es = _run_steps(w, 3, dev)
    assert eo <= tol_for(torch.bfloat16), eo
    assert es <= tol_for(torch.bfloat16), es


@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 64), (128, 128), (32, 128)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decode_shapes(dk, dv, dtype):
    dev = need_gpu()
    w = inputs.Workload("decode_small", "decode", H=3, dk=dk, dv=dv, dtype=dtype, B=5, s0_std=0.02)
    eo, es = _run_steps(w, 4, dev, seed=dk + dv)
    assert eo <= tol_for(dtype), eo
    assert es <= tol_for(dtype), es


def test_decode_matches_prefill_of_same_tokens():
    """n decode steps == prefill of the same n tokens (GPU vs GPU, fp32)."""
    dev = need_gpu()
    w = inputs.Workload("p8", "prefill", H=2, dk=64, dv=64, dtype=torch.float32, chunk=16, T=23, B=1, s0_std=0.02)
    d = inputs.make_prefill(w, device=dev, seed=3)
    O, Sf = kda.kda_prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S0=d["S0"],
                            cu_seqlens=d["cu_seqlens"], cu_seqlens_host=d["cu_seqlens_host"], chunk=16)
    S = d["S0"].clone()
    outs = []
    for t in range(23):
        sl = slice(t, t + 1)
        outs.append(kda.kda_decode(d["q"][sl], d["k"][sl], d["v"][sl], d["log_alpha"][sl], d["beta"][sl], S))
    o = torch.cat(outs)
    assert rel_err(o, O.double().cpu().numpy()) < 1e-5
    assert rel_err(S, Sf.double().cpu().numpy()) < 1e-5
