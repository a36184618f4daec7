"""Chunked prefill: CUDA kernels vs the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import kimi_delta_attention_chunked_gb300 as kda
from kimi_delta_attention_chunked_gb300 import inputs
from _gpu import need_gpu, rel_err, tol_for

pytestmark = pytest.mark.gpu


def run_case(w, dev, lengths=None, seed=0, heads=None, host_cu=True, check=True, alias_state=False):
    d = inputs.make_prefill(w, device=dev, seed=seed, lengths=lengths)
    S0 = d["S0"]
    kw = {}
    if alias_state and S0 is not None:
        state = S0.clone()                     # S0 and S_final are the same buffer
        kw["S_final"] = state
        S_in = state
    else:
        S_in = S0
    O, Sf = kda.kda_prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S0=S_in,
                            cu_seqlens=d["cu_seqlens"], cu_seqlens_host=d["cu_seqlens_host"] if host_cu else None,
                            chunk=w.chunk, **kw)
    torch.cuda.synchronize()
    assert kda.kda_get_last_device_status() == 0
    if not check:
        return d, O, Sf, None, None
    h0, h1 = heads if heads else (0, w.H)
    sl = slice(h0, h1)
    s0 = None if S0 is None else S0[:, sl].contiguous()
    O_ref, Sf_ref = oracle.prefill(d["q"][:, sl].contiguous(), d["k"][:, sl].contiguous(), d["v"][:, sl].contiguous(),
                                   d["log_alpha"][:, sl].contiguous(), d["beta"][:, sl].contiguous(),
                                   cu_seqlens=d["cu_seqlens_host"], S0=s0)
    eo = rel_err(O[:, sl], O_ref)
    es = rel_err(Sf[:, sl], Sf_ref)
    print(f"PARITY {w.name} dtype={w.dtype} lengths={lengths if lengths else d['lengths'][:3]} heads={h0}:{h1} "
          f"O={eo:.3e} S={es:.3e}")
    return d, O, Sf, eo, es


# ------------------------------------------------------------- CUDA-core path
def test_tiny_fp32_workload():
    """B=1, H=2, T=64, d=32, chunk 16, fp32: the 1e-4 correctness case."""
    dev = need_gpu()
    w = inputs.WORKLOADS["tiny_fp32_T64_H2_D32"]
    _, _, _, eo, es = run_case(w, dev)
    assert eo <= 1e-4 and es <= 1e-4, (eo, es)


@pytest.mark.parametrize("dk,dv,chunk", [(32, 32, 16), (64, 32, 32), (128, 64, 64), (32, 128, 16), (64, 64, 64)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_simt_path_varlen(dk, dv, chunk, dtype):
    """Ragged varlen batches (empty, shorter than a chunk, several chunks + tail)."""
    dev = need_gpu()
    w = inputs.Workload("simt", "prefill", H=3, dk=dk, dv=dv, dtype=dtype, chunk=chunk, s0_std=0.02)
    _, _, _, eo, es = run_case(w, dev, lengths=[0, 1, chunk - 1, 2 * chunk + 5, 3 * chunk], seed=dk + chunk)
    assert eo <= tol_for(dtype), eo
    assert es <= tol_for(dtype), es


def test_chunk_size_invariance_fp32():
    """The chunk form is exact for any chunk size: C = 16, 32, 64 agree (fp32)."""
    dev = need_gpu()
    outs = []
    for C in (16, 32, 64):
        w = inputs.Workload("inv", "prefill", H=2, dk=64, dv=64, dtype=torch.float32, chunk=C, s0_std=0.02)
        d, O, Sf, _, _ = run_case(w, dev, lengths=[150, 37], seed=5, check=False)
        outs.append((O.double().cpu().numpy(), Sf.double().cpu().numpy()))
    for O, Sf in outs[1:]:
        assert rel_err(torch.from_numpy(O), outs[0][0]) < 1e-5
        assert rel_err(torch.from_numpy(Sf), outs[0][1]) < 1e-5


# ------------------------------------------------------------- tensor-core path
TC = dict(H=4, dk=128, dv=128, dtype=torch.bfloat16, chunk=64)


@pytest.mark.parametrize("lengths", [[1], [17], [64], [65], [200], [64 * 5], [0, 130, 1, 64, 63, 129]])
def test_tc_path_lengths(lengths):
    dev = need_gpu()
    w = inputs.Workload("tc", "prefill", s0_std=0.02, **TC)
    _, _, _, eo, es = run_case(w, dev, lengths=lengths, seed=len(lengths) + sum(lengths))
    assert eo <= 5e-3, eo
    assert es <= 5e-3, es


def test_tc_path_zero_state_and_device_only_cu_seqlens():
    dev = need_gpu()
    w = inputs.Workload("tc", "prefill", **TC)
    _, _, _, eo, es = run_case(w, dev, lengths=[300, 77, 640], seed=11, host_cu=False)
    assert eo <= 5e-3 and es <= 5e-3, (eo, es)


@pytest.mark.parametrize("host_cu", [True, False])
def test_tc_state_pass_longest_sequences_first(host_cu):
    """More state-pass CTAs than SMs over sequences of different lengths (32
    heads x 7 sequences, one of them empty): the CTAs are launched in the
    order of their sequence's length, ranked on the device (also from a
    device-only cu_seqlens); every sequence's rows and final state still come
    out in place."""
    dev = need_gpu()
    w = inputs.Workload("tc", "prefill", H=32, dk=128, dv=128, dtype=torch.bfloat16, chunk=64, s0_std=0.02)
    _, _, _, eo, es = run_case(w, dev, lengths=[300, 77, 0, 1000, 64, 1000, 5], seed=19, heads=(0, 3),
                               host_cu=host_cu)
    assert eo <= 5e-3 and es <= 5e-3, (eo, es)


def test_tc_path_equal_lengths_without_cu_seqlens():
    """cu_seqlens = NULL: n_seq = 1 sequence covering all tokens."""
    dev = need_gpu()
    w = inputs.Workload("tc", "prefill", T=333, B=1, **TC)
    d = inputs.make_prefill(w, device=dev, seed=12)
    O, Sf = kda.kda_prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"])
    O_ref, Sf_ref = oracle.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"])
    assert rel_err(O, O_ref) <= 5e-3
    assert rel_err(Sf, Sf_ref) <= 5e-3


@pytest.mark.parametrize("dtype,dim,chunk", [(torch.bfloat16, 128, 64), (torch.float32, 32, 16)],
                         ids=["tensor_cores", "cuda_cores"])
def test_all_sequences_empty(dtype, dim, chunk):
    """Every sequence empty (T_total = 0): no output rows, and each S_final is
    its S0 bit for bit (no chunk touches the state)."""
    dev = need_gpu()
    w = inputs.Workload("empty", "prefill", H=4, dk=dim, dv=dim, dtype=dtype, chunk=chunk, s0_std=0.02)
    d = inputs.make_prefill(w, device=dev, seed=3, lengths=[0, 0, 0])
    O, Sf = kda.kda_prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S0=d["S0"],
                            cu_seqlens=d["cu_seqlens"], cu_seqlens_host=d["cu_seqlens_host"], chunk=chunk)
    torch.cuda.synchronize()
    assert kda.kda_get_last_device_status() == 0
    assert O.shape == (0, 4, dim)
    assert torch.equal(Sf, d["S0"])


def test_tc_state_aliasing():
    dev = need_gpu()
    w = inputs.Workload("tc", "prefill", s0_std=0.02, **TC)
    _, _, _, eo, es = run_case(w, dev, lengths=[100, 250], seed=13, alias_state=True)
    assert eo <= 5e-3 and es <= 5e-3, (eo, es)


def test_tc_split_prefill_equals_one_prefill():
    """Prefill of T1 then T2 from the carried state == one prefill of T1 + T2."""
    dev = need_gpu()
    w = inputs.Workload("tc", "prefill", T=448, B=1, s0_std=0.02, **TC)
    d = inputs.make_prefill(w, device=dev, seed=14)
    a = lambda x, s: x[s].contiguous()
    O, Sf = kda.kda_prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S0=d["S0"])
    s1, s2 = slice(0, 192), slice(192, 448)
    O1, S1 = kda.kda_prefill(a(d["q"], s1), a(d["k"], s1), a(d["v"], s1), a(d["log_alpha"], s1), a(d["beta"], s1),
                             S0=d["S0"])
    O2, S2 = kda.kda_prefill(a(d["q"], s2), a(d["k"], s2), a(d["v"], s2), a(d["log_alpha"], s2), a(d["beta"], s2),
                             S0=S1)
    assert rel_err(torch.cat([O1, O2]), O.double().cpu().numpy()) < 5e-3
    assert rel_err(S2, Sf.double().cpu().numpy()) < 5e-3


@pytest.mark.parametrize("H,lengths", [(17, [64 * 1024 + 17]), (8, [70001, 300, 0, 66000])],
                         ids=["17_heads", "varlen_8_heads"])
def test_tc_overlapped_slices(H, lengths):
    """Long sequences whose state pass leaves at least half of the SMs free (17
    heads: 34 state-pass CTAs, too many for the segment scan; a varlen batch at
    8 heads): the prep of later chunk slices runs beside the state pass of
    earlier ones, its CTAs drawing items from a counter on the SMs the state
    pass does not keep; the state crosses slice borders."""
    dev = need_gpu()
    w = inputs.Workload("tc", "prefill", H=H, dk=128, dv=128, dtype=torch.bfloat16, chunk=64, s0_std=0.02)
    _, _, _, eo, es = run_case(w, dev, lengths=lengths, seed=15, heads=(H - 2, H))
    assert eo <= 5e-3 and es <= 5e-3, (lengths, eo, es)


def test_tc_overlapped_slices_long_sequence_32_heads():
    """A long sequence at 32 heads (64 state-pass CTAs, a third of the SMs free
    at most): the prep of later chunk slices runs beside the state pass of
    earlier ones on the SMs it leaves free; a ragged tail and a random S0."""
    dev = need_gpu()
    w = inputs.Workload("tc", "prefill", H=32, dk=128, dv=128, dtype=torch.bfloat16, chunk=64, s0_std=0.02)
    _, _, _, eo, es = run_case(w, dev, lengths=[64 * 1024 + 37], seed=18, heads=(29, 31))
    assert eo <= 5e-3 and es <= 5e-3, (eo, es)


@pytest.mark.parametrize("host_cu", [True, False])
def test_tc_segment_scan_few_heads(host_cu):
    """Two heads and long sequences: each sequence is cut into segments of 16
    chunks; pass 1 gives every segment's affine map, a scan gives its starting
    state, pass 3 its outputs.  Ragged tails, an empty sequence, random S0, and
    device-only lengths."""
    dev = need_gpu()
    w = inputs.Workload("tc", "prefill", H=2, dk=128, dv=128, dtype=torch.bfloat16, chunk=64, s0_std=0.02)
    for lengths in ([64 * 200 + 37], [5000, 64, 0, 3001], [64 * 64]):
        _, _, _, eo, es = run_case(w, dev, lengths=lengths, seed=16, host_cu=host_cu)
        assert eo <= 5e-3 and es <= 5e-3, (lengths, eo, es)


def test_tc_segment_scan_equal_lengths():
    """cu_seqlens = NULL (no chunk table): one sequence of 8320 tokens, one head,
    random S0, split into segments."""
    dev = need_gpu()
    w = inputs.Workload("tc", "prefill", T=8320, B=1, H=1, dk=128, dv=128, dtype=torch.bfloat16, chunk=64,
                        s0_std=0.02)
    d = inputs.make_prefill(w, device=dev, seed=17)
    O, Sf = kda.kda_prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S0=d["S0"])
    torch.cuda.synchronize()
    assert kda.kda_get_last_device_status() == 0
    O_ref, Sf_ref = oracle.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S0=d["S0"])
    assert rel_err(O, O_ref) <= 5e-3
    assert rel_err(Sf, Sf_ref) <= 5e-3


# ------------------------------------------------------------- full-size workloads
def test_full_prefill_8k():
    """B=1, H=32, T=8192, d=128, chunk 64, bf16: every output vs the oracle."""
    dev = need_gpu()
    _, _, _, eo, es = run_case(inputs.WORKLOADS["prefill_bf16_T8192_H32_D128"], dev)
    assert eo <= 5e-3 and es <= 5e-3, (eo, es)


def _oracle_heads(d, heads):
    """The oracle on the listed heads only (gathered into a contiguous batch),
    so that large workloads are compared head group by head group."""
    idx = torch.tensor(list(heads), device=d["q"].device)
    g = lambda x: None if x is None else x.index_select(1, idx).contiguous()
    return oracle.prefill(g(d["q"]), g(d["k"]), g(d["v"]), g(d["log_alpha"]), g(d["beta"]),
                          cu_seqlens=d["cu_seqlens_host"], S0=g(d["S0"]))


def test_full_varlen_all_heads():
    """8 packed sequences of 1K..32K tokens with random S0: all 32 heads vs the
    oracle, O and every final state, compared eight heads at a time."""
    dev = need_gpu()
    w = inputs.WORKLOADS["varlen_bf16_8seq_1K_32K_H32_D128"]
    d, O, Sf, _, _ = run_case(w, dev, check=False)
    worst_o = worst_s = 0.0
    for h0 in range(0, w.H, 8):
        heads = range(h0, h0 + 8)
        O_ref, Sf_ref = _oracle_heads(d, heads)
        worst_o = max(worst_o, rel_err(O[:, h0:h0 + 8], O_ref))
        worst_s = max(worst_s, rel_err(Sf[:, h0:h0 + 8], Sf_ref))
    print(f"PARITY {w.name} lengths={d['lengths']} all heads O={worst_o:.3e} S={worst_s:.3e}")
    assert worst_o <= 5e-3 and worst_s <= 5e-3, (worst_o, worst_s)


@pytest.mark.slow
def test_full_long_context_sampled_heads():
    """T = 1,048,576, H = 32, strong decay: four heads spread over 0..31 vs the
    oracle, every output and the final state."""
    dev = need_gpu()
    w = inputs.WORKLOADS["long_bf16_T1M_H32_D128"]
    d, O, Sf, _, _ = run_case(w, dev, check=False)
    heads = (0, 7, 19, 31)
    O_ref, Sf_ref = _oracle_heads(d, heads)
    idx = torch.tensor(heads, device=dev)
    eo = rel_err(O.index_select(1, idx), O_ref)
    es = rel_err(Sf.index_select(1, idx), Sf_ref)
    print(f"PARITY {w.name} heads={heads} O={eo:.3e} S={es:.3e}")
    assert eo <= 5e-3 and es <= 5e-3, (eo, es)
