"""The debug library (libkda_debug.so, built with KDA_DEBUG) on the GPU.

Its extra checks (include/kda.h, kda_debug_build): a pass over log_alpha
before each call that records KDA_ERR_PRECONDITION when a value leaves the
log-decay bound [-5, 0] of "LLM architecture at trillion scale", section "The
KDA update, in plain words", and device checks of the workspace indices the
tensor-core kernels derive from the call's lengths.  An out-of-range log-decay
only computes less accurately (nothing faults), so feeding one is safe.
Checked through the C ABI of each library: the debug library flags such an
input and the release library does not; on valid inputs the debug library
reports KDA_OK and returns the release library's results bit for bit."""
import ctypes

import pytest
import torch

from kimi_delta_attention_chunked_gb300 import _lib, inputs
from _gpu import need_gpu

pytestmark = pytest.mark.gpu

P = ctypes.c_void_p


def _prefill(lib, d, H, dk, O, Sf, ws, stream):
    T = d["T"]
    host = (ctypes.c_int32 * len(d["cu_seqlens_host"]))(*d["cu_seqlens_host"])
    dt = _lib.KDA_BF16 if d["q"].dtype == torch.bfloat16 else _lib.KDA_FP32
    return lib.kda_prefill(P(d["q"].data_ptr()), P(d["k"].data_ptr()), P(d["v"].data_ptr()),
                           P(d["log_alpha"].data_ptr()), P(d["beta"].data_ptr()), P(d["S0"].data_ptr()),
                           P(d["cu_seqlens"].data_ptr()), host, len(d["lengths"]), T, H, dk, dk, 64, dt,
                           P(O.data_ptr()), P(Sf.data_ptr()), P(ws.data_ptr()) if ws is not None else None,
                           0 if ws is None else ws.numel(), P(stream.cuda_stream))


@pytest.mark.parametrize("dk", [128, 64], ids=["tensor_core", "cuda_core"])
def test_debug_library_flags_log_decay_outside_its_bound(dk):
    dev = need_gpu()
    rel, dbg = _lib.load(), _lib.load_debug()
    assert dbg.kda_debug_build() == 1 and rel.kda_debug_build() == 0
    H = 2
    w = inputs.Workload("dbg", "prefill", H=H, dk=dk, dv=dk, dtype=torch.bfloat16, chunk=64, s0_std=0.02)
    d = inputs.make_prefill(w, device=dev, seed=51, lengths=[200, 77])
    stream = torch.cuda.current_stream(dev)
    need = rel.kda_prefill_workspace_size(2, d["T"], H, dk, dk, 64, _lib.KDA_BF16)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev) if need else None
    outs = {}
    for name, lib in (("release", rel), ("debug", dbg)):
        O = torch.empty_like(d["v"])
        Sf = torch.empty_like(d["S0"])
        assert _prefill(lib, d, H, dk, O, Sf, ws, stream) == _lib.KDA_OK
        assert lib.kda_get_last_device_status(P(stream.cuda_stream)) == _lib.KDA_OK, name
        outs[name] = (O, Sf)
    # valid inputs: the checks change nothing
    assert torch.equal(outs["debug"][0], outs["release"][0])
    assert torch.equal(outs["debug"][1], outs["release"][1])
    # one value below -5 and one above 0
    d["log_alpha"][5, 1, 3] = -6.5
    d["log_alpha"][150, 0, 7] = 0.25
    O = torch.empty_like(d["v"])
    Sf = torch.empty_like(d["S0"])
    assert _prefill(rel, d, H, dk, O, Sf, ws, stream) == _lib.KDA_OK
    assert rel.kda_get_last_device_status(P(stream.cuda_stream)) == _lib.KDA_OK      # unchecked in release
    assert _prefill(dbg, d, H, dk, O, Sf, ws, stream) == _lib.KDA_OK
    assert dbg.kda_get_last_device_status(P(stream.cuda_stream)) == _lib.KDA_ERR_PRECONDITION
    assert dbg.kda_get_last_device_status(P(stream.cuda_stream)) == _lib.KDA_OK      # reading clears it


def test_debug_library_checks_decode_inputs():
    dev = need_gpu()
    dbg = _lib.load_debug()
    w = inputs.Workload("dbg_dec", "decode", H=3, dk=128, dv=128, dtype=torch.bfloat16, B=4, s0_std=0.02)
    dd = inputs.make_decode(w, device=dev, seed=52)
    stream = torch.cuda.current_stream(dev)
    o = torch.empty_like(dd["v"][0])

    def step():
        S = dd["S"].clone()
        st = dbg.kda_decode(P(dd["q"][0].data_ptr()), P(dd["k"][0].data_ptr()), P(dd["v"][0].data_ptr()),
                            P(dd["log_alpha"][0].data_ptr()), P(dd["beta"][0].data_ptr()), P(S.data_ptr()),
                            4, 3, 128, 128, _lib.KDA_BF16, P(o.data_ptr()), P(stream.cuda_stream))
        assert st == _lib.KDA_OK
        return dbg.kda_get_last_device_status(P(stream.cuda_stream))

    assert step() == _lib.KDA_OK
    dd["log_alpha"][0][2, 1, 100] = float("nan")
    assert step() == _lib.KDA_ERR_PRECONDITION
