"""State checkpoints of kda_prefill_ckpt vs the fp64 oracle run on each prefix.

Checkpoint m of a sequence is the state after its first m * ckpt_every tokens;
the oracle computes it as the final state of that prefix (token loop)."""
import numpy as np
import pytest
import torch

import oracle
import kimi_delta_attention_chunked_gb300 as kda
from kimi_delta_attention_chunked_gb300 import inputs
from _gpu import need_gpu, rel_err, tol_for

pytestmark = pytest.mark.gpu


def oracle_checkpoints(d, every, heads):
    """fp64 checkpoints [n_ckpt, heads, dk, dv] by running the oracle on every
    checkpointed prefix of every sequence in one varlen call."""
    sl = slice(*heads)
    bounds = [int(x) for x in d["cu_seqlens_host"]]
    S0 = d["S0"]
    idx, cu, s0 = [], [0], []
    for n in range(len(bounds) - 1):
        bos, ln = bounds[n], bounds[n + 1] - bounds[n]
        for m in range(1, ln // every + 1):
            idx.append(torch.arange(bos, bos + m * every))
            cu.append(cu[-1] + m * every)
            if S0 is not None:
                s0.append(S0[n, sl].cpu())
    if not idx:
        return None
    ix = torch.cat(idx)
    pick = lambda t: t[ix][:, sl].contiguous()
    _, S_ref = oracle.prefill(pick(d["q"].cpu()), pick(d["k"].cpu()), pick(d["v"].cpu()),
                              pick(d["log_alpha"].cpu()), pick(d["beta"].cpu()), cu_seqlens=cu,
                              S0=torch.stack(s0) if s0 else None)
    return S_ref


def run_ckpt(w, dev, lengths, every, seed=0, heads=None, host_cu=True, one_seq=False):
    d = inputs.make_prefill(w, device=dev, seed=seed, lengths=lengths)
    cu = None if one_seq else d["cu_seqlens"]
    S0 = d["S0"][:1] if (one_seq and d["S0"] is not None) else d["S0"]
    n_ck = kda.checkpoint_count(d["lengths"], every)
    ckpt = torch.full((max(n_ck, 1), w.H, w.dk, w.dv), float("nan"), device=dev)[:n_ck]
    O, Sf, ck = kda.kda_prefill_ckpt(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], every, S0=S0,
                                     cu_seqlens=cu, cu_seqlens_host=d["cu_seqlens_host"] if (host_cu and cu is not None)
                                     else None, chunk=w.chunk, ckpt=ckpt)
    O2, Sf2 = kda.kda_prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S0=S0, cu_seqlens=cu,
                              cu_seqlens_host=d["cu_seqlens_host"] if cu is not None else None, chunk=w.chunk)
    torch.cuda.synchronize()
    assert kda.kda_get_last_device_status() == 0
    # the same kernels run: outputs identical to kda_prefill's
    assert torch.equal(O, O2) and torch.equal(Sf, Sf2)
    heads = heads or (0, w.H)
    ref = oracle_checkpoints(d, every, heads)
    if ref is None:
        assert n_ck == 0
        return 0.0
    e = rel_err(ck[:, heads[0]:heads[1]], ref)
    print(f"PARITY ckpt {w.name} dtype={w.dtype} lengths={d['lengths'][:6]} every={every} n_ckpt={n_ck} "
          f"heads={heads[0]}:{heads[1]} S={e:.3e}")
    return e


TC = dict(H=4, dk=128, dv=128, dtype=torch.bfloat16, chunk=64)


@pytest.mark.parametrize("every", [64, 192])
def test_tc_ckpt_varlen(every):
    """Tensor-core path, ragged batch: lengths below, at and above multiples."""
    dev = need_gpu()
    w = inputs.Workload("tc_ckpt", "prefill", s0_std=0.02, **TC)
    e = run_ckpt(w, dev, [0, 300, 576, 1000, 64, 191], every, seed=11)
    assert e <= tol_for(w.dtype), e


def test_tc_ckpt_device_only_lengths():
    """Lengths only on the device: checkpoint indices come from the kernel's own prefix sum."""
    dev = need_gpu()
    w = inputs.Workload("tc_ckpt_dev", "prefill", s0_std=0.02, **TC)
    e = run_ckpt(w, dev, [130, 0, 640, 257], 128, seed=12, host_cu=False)
    assert e <= tol_for(w.dtype), e


def test_tc_ckpt_one_sequence_narrow_slices():
    """One sequence, few heads: the state pass runs over 32-column slices."""
    dev = need_gpu()
    w = inputs.Workload("tc_ckpt_one", "prefill", s0_std=0.02, **TC)
    e = run_ckpt(w, dev, [4096], 256, seed=13, one_seq=True, heads=(0, 2))
    assert e <= tol_for(w.dtype), e


def test_tc_ckpt_long_sequence_overlapped_slices():
    """A long sequence (1027 chunks, 2 heads; checkpoints keep it off the
    segment scan): the prep of later chunk slices runs beside the state pass,
    which carries the state across slice borders, and checkpoints fall near
    them."""
    dev = need_gpu()
    w = inputs.Workload("tc_ckpt_long", "prefill", H=2, dk=128, dv=128, dtype=torch.bfloat16, chunk=64,
                        s0_std=0.02)
    e = run_ckpt(w, dev, [64 * 1027], 8192, seed=14, one_seq=True)
    assert e <= tol_for(w.dtype), e


def test_tc_ckpt_many_heads_longest_sequences_first():
    """More state-pass CTAs than SMs (32 heads x 7 sequences): the CTAs run in
    the order of their sequence's length, and each writes its own sequence's
    checkpoints."""
    dev = need_gpu()
    w = inputs.Workload("tc_ckpt_many", "prefill", H=32, dk=128, dv=128, dtype=torch.bfloat16, chunk=64,
                        s0_std=0.02)
    e = run_ckpt(w, dev, [300, 77, 0, 1000, 64, 1000, 5], 64, seed=15, heads=(0, 2))
    assert e <= tol_for(w.dtype), e


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dk,dv,chunk,every", [(32, 32, 16, 32), (64, 64, 32, 32), (128, 64, 64, 128)])
def test_simt_ckpt_varlen(dtype, dk, dv, chunk, every):
    dev = need_gpu()
    w = inputs.Workload("simt_ckpt", "prefill", H=3, dk=dk, dv=dv, dtype=dtype, chunk=chunk, s0_std=0.02)
    e = run_ckpt(w, dev, [0, every - 1, every, 3 * every + 5, 2 * chunk + 1], every, seed=dk + every)
    assert e <= tol_for(dtype), e


def test_simt_ckpt_equal_lengths_fp32():
    dev = need_gpu()
    w = inputs.Workload("simt_ckpt_one", "prefill", H=2, dk=64, dv=64, dtype=torch.float32, chunk=16,
                        s0_std=0.02)
    e = run_ckpt(w, dev, [320], 64, seed=3, one_seq=True)
    assert e <= tol_for(w.dtype), e
