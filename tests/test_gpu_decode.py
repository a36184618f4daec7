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


@pytest.mark.slow
def test_decode_1000_consecutive_steps():
    """The decode workload as benchmarked: 256 sequences x 32 heads, 1000
    consecutive in-place steps, each with a fresh token set.  Every head of
    eight sequences spread over the batch (256 (sequence, head) chains) is
    checked against the oracle: o of every step, and the state after step 1000.
    The oracle runs each chain's 1000 tokens as one sequence from the same
    initial state (decode is the recurrence one token at a time)."""
    dev = need_gpu()
    w = inputs.WORKLOADS["decode_bf16_N256_H32_D128"]
    steps = 1000
    d = inputs.make_decode(w, device=dev, seed=0, n_token_sets=steps)
    sel = torch.arange(0, w.B, w.B // 8, device=dev)[:8]          # 8 sequences x all 32 heads
    S = d["S"].clone()
    o_sel = []
    for t in range(steps):
        o = kda.kda_decode(d["q"][t], d["k"][t], d["v"][t], d["log_alpha"][t], d["beta"][t], S)
        o_sel.append(o.index_select(0, sel))
    torch.cuda.synchronize()
    assert kda.kda_get_last_device_status() == 0
    # oracle input: chain n's tokens are its rows of the 1000 token sets, in order
    pack = lambda xs: torch.stack([x.index_select(0, sel) for x in xs], dim=1).reshape(
        (len(sel) * steps,) + tuple(xs[0].shape[1:])).contiguous()
    cu = [i * steps for i in range(len(sel) + 1)]
    O_ref, S_ref = oracle.prefill(pack(d["q"]), pack(d["k"]), pack(d["v"]), pack(d["log_alpha"]),
                                  pack(d["beta"]), cu_seqlens=cu, S0=d["S"].index_select(0, sel))
    o_gpu = torch.stack(o_sel, dim=1).double().cpu().numpy()           # [8, steps, H, dv]
    O_ref = O_ref.reshape(o_gpu.shape)
    assert np.all(np.isfinite(o_gpu))
    # the bar per step (each step is one call): max |o - o_ref| / max |o_ref| over its outputs
    eo = max(float(np.max(np.abs(o_gpu[:, t] - O_ref[:, t]))) / float(np.max(np.abs(O_ref[:, t])))
             for t in range(steps))
    es = rel_err(S.index_select(0, sel), S_ref)
    print(f"PARITY decode 1000 steps, 256 chains: o={eo:.3e} S={es:.3e}")
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


@pytest.mark.parametrize("K", [1, 3, 8, 16])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_verify_multi_token(K, dtype):
    """K proposed tokens per sequence (16 = the most the kernel stages): every
    output vs the oracle; the state is committed after commit_len[n] tokens
    (0 .. K, drawn per sequence)."""
    dev = need_gpu()
    N, H, D = 16, 4, 128
    w = inputs.Workload("verify", "prefill", H=H, dk=D, dv=D, dtype=dtype, chunk=64, T=K, B=N, s0_std=0.02)
    d = inputs.make_prefill(w, device=dev, seed=K, lengths=[K] * N)
    rs = lambda x, last: x.view(N, K, H, last).contiguous()
    q, k, v, g = rs(d["q"], D), rs(d["k"], D), rs(d["v"], D), rs(d["log_alpha"], D)
    b = d["beta"].view(N, K, H).contiguous()
    S = d["S0"].clone()
    commit = torch.tensor([(7 * n) % (K + 1) for n in range(N)], dtype=torch.int32, device=dev)
    o = kda.kda_decode_multi(q, k, v, g, b, S, commit_len=commit)
    torch.cuda.synchronize()
    assert kda.kda_get_last_device_status() == 0
    O_ref, _ = oracle.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], cu_seqlens=d["cu_seqlens_host"],
                              S0=d["S0"])
    assert rel_err(o.view(N * K, H, D), O_ref) <= tol_for(dtype)
    for n in range(N):
        c = int(commit[n])
        if c == 0:
            ref = d["S0"][n].double().cpu().numpy()
        else:
            sl = slice(n * K, n * K + c)
            _, Sf = oracle.prefill(d["q"][sl], d["k"][sl], d["v"][sl], d["log_alpha"][sl], d["beta"][sl],
                                   S0=d["S0"][n:n + 1])
            ref = Sf[0]
        assert rel_err(S[n], ref) <= tol_for(dtype), n


@pytest.mark.parametrize("dk,dv", [(32, 32), (32, 128), (64, 128), (128, 64)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_verify_shapes(dk, dv, dtype):
    """The verify kernel at the other head dims (one instantiation each): outputs
    and the state after all K tokens vs the oracle."""
    dev = need_gpu()
    N, K, H = 8, 5, 2
    w = inputs.Workload("verify4", "prefill", H=H, dk=dk, dv=dv, dtype=dtype, chunk=64, T=K, B=N, s0_std=0.02)
    d = inputs.make_prefill(w, device=dev, seed=dk + dv, lengths=[K] * N)
    q, k, g = (d[n].view(N, K, H, dk).contiguous() for n in ("q", "k", "log_alpha"))
    v = d["v"].view(N, K, H, dv).contiguous()
    b = d["beta"].view(N, K, H).contiguous()
    S = d["S0"].clone()
    o = kda.kda_decode_multi(q, k, v, g, b, S)
    torch.cuda.synchronize()
    assert kda.kda_get_last_device_status() == 0
    O_ref, S_ref = oracle.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], cu_seqlens=d["cu_seqlens_host"],
                                  S0=d["S0"])
    assert rel_err(o.view(N * K, H, dv), O_ref) <= tol_for(dtype)
    assert rel_err(S, S_ref) <= tol_for(dtype)


def test_verify_outputs_only_then_commit():
    """The two-call pattern: outputs with nothing committed, then a commit-only call."""
    dev = need_gpu()
    N, K, H, D = 8, 5, 2, 64
    w = inputs.Workload("verify2", "prefill", H=H, dk=D, dv=D, dtype=torch.float32, chunk=64, T=K, B=N, s0_std=0.02)
    d = inputs.make_prefill(w, device=dev, seed=99, lengths=[K] * N)
    rs = lambda x: x.view(N, K, H, D).contiguous()
    b = d["beta"].view(N, K, H).contiguous()
    S = d["S0"].clone()
    zero = torch.zeros(N, dtype=torch.int32, device=dev)
    o = kda.kda_decode_multi(rs(d["q"]), rs(d["k"]), rs(d["v"]), rs(d["log_alpha"]), b, S, commit_len=zero)
    assert torch.equal(S, d["S0"])                    # nothing committed
    acc = torch.tensor([K, 0, 1, 2, 3, 4, K, 1], dtype=torch.int32, device=dev)
    assert kda.kda_decode_multi(rs(d["q"]), rs(d["k"]), rs(d["v"]), rs(d["log_alpha"]), b, S, commit_len=acc,
                                want_o=False) is None
    for n in range(N):
        c = int(acc[n])
        if c:
            sl = slice(n * K, n * K + c)
            _, Sf = oracle.prefill(d["q"][sl], d["k"][sl], d["v"][sl], d["log_alpha"][sl], d["beta"][sl],
                                   S0=d["S0"][n:n + 1])
            assert rel_err(S[n], Sf[0]) <= 1e-4
        else:
            assert torch.equal(S[n], d["S0"][n])


def test_verify_unaligned_inputs_take_the_scalar_staging():
    """Inputs at an odd element offset (2 bytes past an aligned start): the
    results are the same bits as from aligned copies of the same inputs, and
    match the oracle."""
    dev = need_gpu()
    N, K, H, D = 8, 8, 4, 128
    w = inputs.Workload("verify3", "prefill", H=H, dk=D, dv=D, dtype=torch.bfloat16, chunk=64, T=K, B=N, s0_std=0.02)
    d = inputs.make_prefill(w, device=dev, seed=5, lengths=[K] * N)
    rs = lambda x: x.view(N, K, H, D).contiguous()

    def shifted(x):                                   # same values, one element past an aligned start
        buf = torch.empty(x.numel() + 1, dtype=x.dtype, device=dev)
        buf[1:].copy_(x.reshape(-1))
        return buf[1:].view(x.shape)

    b = d["beta"].view(N, K, H).contiguous()
    args = [rs(d[n]) for n in ("q", "k", "v", "log_alpha")]
    S1, S2 = d["S0"].clone(), d["S0"].clone()
    o1 = kda.kda_decode_multi(*args, b, S1)
    o2 = kda.kda_decode_multi(*[shifted(a) for a in args], b, S2)
    torch.cuda.synchronize()
    assert kda.kda_get_last_device_status() == 0
    assert torch.equal(o1, o2) and torch.equal(S1, S2)
    O_ref, S_ref = oracle.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], cu_seqlens=d["cu_seqlens_host"],
                                  S0=d["S0"])
    assert rel_err(o2.view(N * K, H, D), O_ref) <= tol_for(torch.bfloat16)
    assert rel_err(S2, S_ref) <= tol_for(torch.bfloat16)
