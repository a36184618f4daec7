"""The Python binding refuses, before anything reaches the C ABI, tensors
whose shapes do not match the sizes it passes (the kernels would index past
them).  CPU tensors suffice: shapes are checked before the device is."""
import pytest
import torch

import kimi_delta_attention_chunked_gb300 as kda
from kimi_delta_attention_chunked_gb300 import _lib, build


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return _lib.load()


def prefill_args(T=70, H=3, dk=32, dv=16, n_seq=2):
    z = lambda *s, dt=torch.float32: torch.zeros(*s, dtype=dt)
    return dict(q=z(T, H, dk), k=z(T, H, dk), v=z(T, H, dv), log_alpha=z(T, H, dk), beta=z(T, H),
                S0=z(n_seq, H, dk, dv), cu_seqlens=torch.tensor([0, 30, T], dtype=torch.int32),
                cu_seqlens_host=[0, 30, T])


def call_prefill(fn=kda.kda_prefill, **kw):
    a = prefill_args()
    a.update(kw)
    return fn(a.pop("q"), a.pop("k"), a.pop("v"), a.pop("log_alpha"), a.pop("beta"), **a)


@pytest.mark.parametrize("fn", [kda.kda_prefill, kda.kda_prefill_noalloc])
def test_prefill_accepts_matching_shapes_up_to_the_device_check(fn):
    with pytest.raises(ValueError, match="must be on"):
        call_prefill(fn)


@pytest.mark.parametrize("name,bad", [
    ("k", (70, 3, 16)), ("v", (69, 3, 16)), ("log_alpha", (70, 3, 31)), ("beta", (70, 2)),
    ("S0", (1, 3, 32, 16)), ("S0", (2, 3, 16, 32)), ("O", (70, 3, 32)), ("S_final", (3, 3, 32, 16)),
])
def test_prefill_refuses_mismatched_shapes(name, bad):
    with pytest.raises(ValueError, match="shape|leading dims"):
        call_prefill(**{name: torch.zeros(*bad)})


def test_prefill_refuses_bad_offsets():
    with pytest.raises(ValueError, match="cu_seqlens_host"):
        call_prefill(cu_seqlens_host=[0, 70])
    with pytest.raises(ValueError, match="cu_seqlens must be"):
        call_prefill(cu_seqlens=torch.tensor([[0, 30, 70]], dtype=torch.int32), cu_seqlens_host=None, S0=None)
    with pytest.raises(ValueError, match="cu_seqlens must be"):
        call_prefill(cu_seqlens=torch.zeros(0, dtype=torch.int32), cu_seqlens_host=None, S0=None)
    with pytest.raises(ValueError, match="dims"):
        call_prefill(q=torch.zeros(70, 3, 2, 16), v=torch.zeros(70, 3, 2, 16))


def test_ckpt_buffer_trailing_dims():
    a = prefill_args()
    with pytest.raises(ValueError, match="ckpt must have shape"):
        kda.kda_prefill_ckpt(a["q"], a["k"], a["v"], a["log_alpha"], a["beta"], 16, S0=a["S0"],
                             cu_seqlens=a["cu_seqlens"], chunk=16, ckpt=torch.zeros(4, 3, 16, 32))


def decode_args(N=5, H=2, dk=64, dv=32):
    z = lambda *s: torch.zeros(*s)
    return [z(N, H, dk), z(N, H, dk), z(N, H, dv), z(N, H, dk), z(N, H), z(N, H, dk, dv)]


def test_decode_shapes():
    with pytest.raises(ValueError, match="must be on"):
        kda.kda_decode(*decode_args())
    for i, bad in [(1, (5, 2, 32)), (2, (4, 2, 32)), (3, (5, 2, 63)), (4, (5,)), (5, (5, 2, 32, 64))]:
        args = decode_args()
        args[i] = torch.zeros(*bad)
        with pytest.raises(ValueError, match="shape|leading dims"):
            kda.kda_decode(*args)
    with pytest.raises(ValueError, match="o must have shape"):
        kda.kda_decode(*decode_args(), o=torch.zeros(5, 2, 64))


def test_verify_shapes():
    N, K, H, dk, dv = 4, 3, 2, 32, 64
    z = lambda *s: torch.zeros(*s)
    args = [z(N, K, H, dk), z(N, K, H, dk), z(N, K, H, dv), z(N, K, H, dk), z(N, K, H), z(N, H, dk, dv)]
    with pytest.raises(ValueError, match="must be on"):
        kda.kda_decode_multi(*args)
    bad = list(args)
    bad[4] = z(N, H)
    with pytest.raises(ValueError, match="beta must have shape"):
        kda.kda_decode_multi(*bad)
    with pytest.raises(ValueError, match="commit_len must have shape"):
        kda.kda_decode_multi(*args, commit_len=torch.zeros(N + 1, dtype=torch.int32))
    with pytest.raises(ValueError, match="o must have shape"):
        kda.kda_decode_multi(*args, o=z(N, K, H, dk))
