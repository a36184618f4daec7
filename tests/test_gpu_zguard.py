"""Writes stay inside the tensors the kernels are given, and parity holds at
the gate's degenerate values.

O, S_final, the decode state and the checkpoint array are handed to the
kernels as views into larger buffers whose margins hold a sentinel: after the
call every margin must be unchanged (parity compares only what lies inside a
tensor and cannot see a write past its end).  The degenerate gates are the
method's special cases: beta = 0 (nothing is written: S_T = Diag(prod alpha)
S0, here under a mild constant decay so that the surviving state stays far
inside fp32's range), beta = 1 (the full delta-rule write) and log alpha = -5
on every channel (the strongest decay the log-decay bound allows, where the
chunk's cumulative log-decay reaches -320 and the staged decay factors reach
their extremes)."""
import math

import pytest
import torch

import oracle
import kimi_delta_attention_chunked_gb300 as kda
from kimi_delta_attention_chunked_gb300 import inputs
from _gpu import need_gpu, rel_err

pytestmark = pytest.mark.gpu

MARGIN = 4096                 # elements on each side; keeps the view 16-byte aligned
SENTINEL = 1234.5


def guarded(shape, dtype, dev, init=None):
    """(buffer, view): the view has ``shape`` and sits between two margins of
    SENTINEL; it starts as ``init`` (or SENTINEL)."""
    n = math.prod(shape)
    buf = torch.full((MARGIN + n + MARGIN,), SENTINEL, dtype=dtype, device=dev)
    view = buf[MARGIN:MARGIN + n].view(shape)
    if init is not None:
        view.copy_(init)
    return buf, view


def margins_intact(buf):
    ref = torch.full((MARGIN,), SENTINEL, dtype=buf.dtype, device=buf.device)
    return torch.equal(buf[:MARGIN], ref) and torch.equal(buf[-MARGIN:], ref)


def prefill_guarded(w, dev, lengths, seed, tol, host_cu=True):
    d = inputs.make_prefill(w, device=dev, seed=seed, lengths=lengths)
    T, n_seq = d["T"], len(lengths)
    ob, O = guarded((T, w.H, w.dv), w.dtype, dev)
    sb, Sf = guarded((n_seq, w.H, w.dk, w.dv), torch.float32, dev)
    kda.kda_prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S0=d["S0"], cu_seqlens=d["cu_seqlens"],
                    cu_seqlens_host=d["cu_seqlens_host"] if host_cu else None, chunk=w.chunk, O=O, S_final=Sf)
    torch.cuda.synchronize()
    assert kda.kda_get_last_device_status() == 0
    assert margins_intact(ob), "a write past O"
    assert margins_intact(sb), "a write past S_final"
    O_ref, S_ref = oracle.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                  cu_seqlens=d["cu_seqlens_host"], S0=d["S0"])
    eo, es = rel_err(O, O_ref), rel_err(Sf, S_ref)
    assert eo <= tol and es <= tol, (eo, es)


# the tensor-core prefill's launch shapes: one state pass over 32-column slices
# (varlen, device-only lengths), the segment scan (2 heads, one long
# sequence), prep slices beside the state pass on two streams (17 heads, one
# sequence of 1025 chunks), and more state-pass CTAs than SMs, launched
# longest sequence first (32 heads, 7 sequences)
TC_CASES = {"tc_varlen": (4, [300, 77, 0, 129, 1]), "tc_device_lengths": (4, [300, 77, 0, 129, 1]),
            "tc_segment_scan": (2, [64 * 40 + 17]), "tc_overlap": (17, [64 * 1024 + 17]),
            "tc_ordered": (32, [300, 77, 0, 1000, 64, 1000, 5])}


@pytest.mark.parametrize("case", list(TC_CASES) + ["simt_fp32"])
def test_prefill_writes_stay_inside(case):
    dev = need_gpu()
    if case.startswith("tc"):
        H, lengths = TC_CASES[case]
        w = inputs.Workload("guard", "prefill", H=H, dk=128, dv=128, dtype=torch.bfloat16, chunk=64, s0_std=0.02)
        prefill_guarded(w, dev, lengths, seed=31, tol=5e-3, host_cu=case != "tc_device_lengths")
    else:
        w = inputs.Workload("guard", "prefill", H=3, dk=64, dv=32, dtype=torch.float32, chunk=32, s0_std=0.02)
        prefill_guarded(w, dev, [70, 5, 0, 33], seed=32, tol=1e-4)


def test_decode_writes_stay_inside():
    dev = need_gpu()
    w = inputs.Workload("guard_dec", "decode", H=3, dk=128, dv=64, dtype=torch.bfloat16, B=7, s0_std=0.02)
    d = inputs.make_decode(w, device=dev, seed=33)
    sb, S = guarded(tuple(d["S"].shape), torch.float32, dev, init=d["S"])
    ob, o = guarded((7, 3, 64), torch.bfloat16, dev)
    kda.kda_decode(d["q"][0], d["k"][0], d["v"][0], d["log_alpha"][0], d["beta"][0], S, o=o)
    torch.cuda.synchronize()
    assert kda.kda_get_last_device_status() == 0
    assert margins_intact(sb) and margins_intact(ob)
    o_ref, S_ref = oracle.decode(d["q"][0], d["k"][0], d["v"][0], d["log_alpha"][0], d["beta"][0], d["S"])
    assert rel_err(o, o_ref) <= 5e-3 and rel_err(S, S_ref) <= 5e-3


def test_checkpoint_writes_stay_inside():
    dev = need_gpu()
    w = inputs.Workload("guard_ck", "prefill", H=2, dk=128, dv=128, dtype=torch.bfloat16, chunk=64, s0_std=0.02)
    lengths, every = [64 * 5 + 3, 128, 63], 64
    d = inputs.make_prefill(w, device=dev, seed=34, lengths=lengths)
    n_ck = kda.checkpoint_count(lengths, every)
    cb, ck = guarded((n_ck, 2, 128, 128), torch.float32, dev)
    O, Sf, _ = kda.kda_prefill_ckpt(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], every, S0=d["S0"],
                                    cu_seqlens=d["cu_seqlens"], cu_seqlens_host=d["cu_seqlens_host"], chunk=64,
                                    ckpt=ck)
    torch.cuda.synchronize()
    assert kda.kda_get_last_device_status() == 0
    assert margins_intact(cb), "a write past the checkpoint array"
    # the last checkpoint of sequence 1 (128 tokens) is its final state
    assert rel_err(ck[5 + 2 - 1], Sf[1].double().cpu().numpy()) <= 1e-4


@pytest.mark.parametrize("gate", ["beta0", "beta1", "decay_max"])
@pytest.mark.parametrize("path", ["tc", "simt_fp32"])
def test_degenerate_gates(gate, path):
    dev = need_gpu()
    if path == "tc":
        w = inputs.Workload("degen", "prefill", H=2, dk=128, dv=128, dtype=torch.bfloat16, chunk=64, s0_std=0.02)
        tol = 5e-3
    else:
        w = inputs.Workload("degen", "prefill", H=2, dk=64, dv=64, dtype=torch.float32, chunk=32, s0_std=0.02)
        tol = 1e-4
    d = inputs.make_prefill(w, device=dev, seed=35, lengths=[300, 77])
    if gate == "beta0":
        # nothing is written, so S only decays: a mild constant decay keeps
        # Diag(prod alpha) S0 far above fp32's range limit over 377 tokens
        d["beta"].zero_()
        d["log_alpha"].fill_(-0.01)
    elif gate == "beta1":
        d["beta"].fill_(1.0)
    else:
        d["log_alpha"].fill_(-5.0)
    O, Sf = kda.kda_prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S0=d["S0"],
                            cu_seqlens=d["cu_seqlens"], cu_seqlens_host=d["cu_seqlens_host"], chunk=w.chunk)
    torch.cuda.synchronize()
    assert kda.kda_get_last_device_status() == 0
    assert torch.isfinite(O.float()).all() and torch.isfinite(Sf).all()
    O_ref, S_ref = oracle.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                  cu_seqlens=d["cu_seqlens_host"], S0=d["S0"])
    eo, es = rel_err(O, O_ref), rel_err(Sf, S_ref)
    print(f"PARITY degenerate {gate} {path}: O={eo:.3e} S={es:.3e}")
    assert eo <= tol and es <= tol, (eo, es)
    if gate == "beta0":
        # nothing written: S_T = Diag(prod alpha) S0 per sequence
        for n, (a, e) in enumerate(zip(d["cu_seqlens_host"][:-1], d["cu_seqlens_host"][1:])):
            decay = torch.exp(d["log_alpha"][a:e].double().sum(0))            # [H, dk]
            expect = (decay[..., None] * d["S0"][n].double()).cpu().numpy()
            assert rel_err(Sf[n], expect) <= tol
