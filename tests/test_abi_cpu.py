"""The C-ABI library loads on a CPU-only host, exports every entry point that
include/kda.h declares, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

import kimi_delta_attention_chunked_gb300 as kda
from kimi_delta_attention_chunked_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"KDA_API\s+[\w\s\*]+?\b(kda_\w+)\s*\(", text)


def test_header_declares_the_api():
    names = declared_functions()
    assert sorted(names) == sorted(_lib.SYMBOLS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    # and nothing that is not declared leaks out as kda_*
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True, text=True).stdout
    exported = sorted(set(re.findall(r"\s(kda_\w+)$", out, re.M)))
    assert exported == sorted(declared_functions())


def test_debug_library_exports_the_same_api():
    """libkda_debug.so (KDA_DEBUG: precondition and device index checks) has
    exactly the release library's entry points, and says which build it is."""
    import subprocess
    build.build()
    dbg = _lib.load_debug()
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_DEBUG_PATH], capture_output=True, text=True).stdout
    assert sorted(set(re.findall(r"\s(kda_\w+)$", out, re.M))) == sorted(declared_functions())
    assert dbg.kda_debug_build() == 1
    assert _lib.load().kda_debug_build() == 0
    # host-side argument checks are the same
    assert dbg.kda_check_wait_timeout(-1, None) == _lib.KDA_ERR_INVALID_ARG


def test_wait_check_rejects_bad_limits_before_launch(lib):
    # checked on the host: nothing is launched (no GPU is needed for this)
    assert lib.kda_check_wait_timeout(-1, None) == _lib.KDA_ERR_INVALID_ARG
    assert lib.kda_check_wait_timeout(1 << 40, None) == _lib.KDA_ERR_INVALID_ARG


def test_status_strings(lib):
    for code in range(8):
        s = kda.kda_status_string(code)
        assert s.startswith("KDA"), s
    assert "unknown" in kda.kda_status_string(99)


def test_workspace_size_is_host_only(lib):
    import torch
    # tensor-core path: (T/C + n_seq) chunk slots x H blocks, plus a small header
    ws1 = kda.kda_prefill_workspace_size(1, 8192, 32, 128, 128, 64, torch.bfloat16)
    ws2 = kda.kda_prefill_workspace_size(1, 8192 + 64, 32, 128, 128, 64, torch.bfloat16)
    block = (ws2 - ws1) // 32                       # one more chunk slot for each of 32 heads
    assert block % 1024 == 0 and 64 * 1024 <= block <= 160 * 1024
    assert ws1 >= (8192 // 64 + 1) * 32 * block
    # the CUDA-core path needs none
    assert kda.kda_prefill_workspace_size(1, 64, 2, 32, 32, 16, torch.float32) == 0
    assert kda.kda_prefill_workspace_size(1, 64, 2, 128, 128, 32, torch.bfloat16) == 0


def _prefill_raw(lib, **kw):
    P = ctypes.c_void_p
    fake = P(0x1000)
    args = dict(q=fake, k=fake, v=fake, g=fake, b=fake, S0=None, cu=None, cuh=None, n_seq=1, T=64, H=2,
                dk=32, dv=32, chunk=16, dt=_lib.KDA_FP32, O=P(0x2000), Sf=None, ws=None, ws_bytes=0, stream=None)
    args.update(kw)
    return lib.kda_prefill(args["q"], args["k"], args["v"], args["g"], args["b"], args["S0"], args["cu"],
                           args["cuh"], args["n_seq"], args["T"], args["H"], args["dk"], args["dv"],
                           args["chunk"], args["dt"], args["O"], args["Sf"], args["ws"], args["ws_bytes"],
                           args["stream"])


def test_prefill_argument_checks(lib):
    E = _lib
    assert _prefill_raw(lib, dk=48) == E.KDA_ERR_UNSUPPORTED
    assert _prefill_raw(lib, dv=256) == E.KDA_ERR_UNSUPPORTED
    assert _prefill_raw(lib, chunk=128) == E.KDA_ERR_UNSUPPORTED
    assert _prefill_raw(lib, dt=7) == E.KDA_ERR_INVALID_ARG
    assert _prefill_raw(lib, H=0) == E.KDA_ERR_INVALID_ARG
    assert _prefill_raw(lib, T=-1) == E.KDA_ERR_INVALID_ARG
    assert _prefill_raw(lib, q=None) == E.KDA_ERR_INVALID_ARG
    assert _prefill_raw(lib, O=None) == E.KDA_ERR_INVALID_ARG
    assert _prefill_raw(lib, O=ctypes.c_void_p(0x1000)) == E.KDA_ERR_INVALID_ARG      # O aliases q
    assert _prefill_raw(lib, n_seq=3, T=64) == E.KDA_ERR_INVALID_ARG                 # 64 % 3 != 0
    assert _prefill_raw(lib, n_seq=0, T=0) == E.KDA_OK                               # nothing to do
    # host cu_seqlens: must start at 0, end at T_total, be non-decreasing
    bad = (ctypes.c_int32 * 3)(0, 40, 30)
    assert _prefill_raw(lib, n_seq=2, cu=ctypes.c_void_p(0x3000), cuh=bad) == E.KDA_ERR_INVALID_ARG
    bad_end = (ctypes.c_int32 * 3)(0, 10, 63)
    assert _prefill_raw(lib, n_seq=2, cu=ctypes.c_void_p(0x3000), cuh=bad_end) == E.KDA_ERR_INVALID_ARG
    # host copy without a device array
    ok = (ctypes.c_int32 * 2)(0, 64)
    assert _prefill_raw(lib, cuh=ok) == E.KDA_ERR_INVALID_ARG
    # tensor-core path: workspace missing / too small / misaligned
    tc = dict(dk=128, dv=128, chunk=64, dt=_lib.KDA_BF16)
    assert _prefill_raw(lib, **tc) == E.KDA_ERR_WORKSPACE
    need = lib.kda_prefill_workspace_size(1, 64, 2, 128, 128, 64, _lib.KDA_BF16)
    assert _prefill_raw(lib, ws=ctypes.c_void_p(0x100000), ws_bytes=need - 1, **tc) == E.KDA_ERR_WORKSPACE
    assert _prefill_raw(lib, ws=ctypes.c_void_p(0x100010), ws_bytes=need, **tc) == E.KDA_ERR_WORKSPACE
    # tensor-core path: token rows move as 16-byte vectors, so unaligned tensors are refused
    ws = dict(ws=ctypes.c_void_p(0x100000), ws_bytes=need, **tc)
    for name in ("q", "k", "v", "g"):
        assert _prefill_raw(lib, **{name: ctypes.c_void_p(0x1008)}, **ws) == E.KDA_ERR_INVALID_ARG, name
    assert _prefill_raw(lib, O=ctypes.c_void_p(0x2008), **ws) == E.KDA_ERR_INVALID_ARG


def test_prefill_ckpt_argument_checks(lib):
    """Checkpoint arguments are checked on the host, before any device work."""
    E = _lib
    P = ctypes.c_void_p
    fake = P(0x1000)

    def call(every=16, ck=P(0x5000), cap=4, n_seq=1, T=64, cu=None, cuh=None, chunk=16):
        return lib.kda_prefill_ckpt(fake, fake, fake, fake, fake, None, cu, cuh, n_seq, T, 2, 32, 32, chunk,
                                    _lib.KDA_FP32, P(0x2000), None, every, ck, cap, None, 0, None)
    assert call(every=0) == E.KDA_ERR_INVALID_ARG
    assert call(every=24) == E.KDA_ERR_INVALID_ARG                 # not a multiple of the chunk
    assert call(cap=-1) == E.KDA_ERR_INVALID_ARG
    assert call(ck=None) == E.KDA_ERR_INVALID_ARG                  # capacity without a buffer
    assert call(ck=P(0x5004)) == E.KDA_ERR_INVALID_ARG             # not 16-byte aligned
    assert call(cap=3) == E.KDA_ERR_INVALID_ARG                    # 64 / 16 = 4 checkpoints needed
    assert call(every=32, cap=1) == E.KDA_ERR_INVALID_ARG
    assert call(every=16, chunk=128) == E.KDA_ERR_UNSUPPORTED
    cuh = (ctypes.c_int32 * 3)(0, 40, 64)                          # 40 // 16 + 24 // 16 = 3
    assert call(n_seq=2, cu=P(0x3000), cuh=cuh, cap=2) == E.KDA_ERR_INVALID_ARG
    assert call(n_seq=0, T=0, cap=0, ck=None) == E.KDA_OK


def test_checkpoint_count():
    assert _lib.checkpoint_count([0, 15, 16, 40, 64], 16) == 0 + 0 + 1 + 2 + 4


def test_decode_argument_checks(lib):
    P = ctypes.c_void_p
    f = P(0x1000)
    S = P(0x4000)
    o = P(0x5000)
    E = _lib
    call = lambda **kw: lib.kda_decode(kw.get("q", f), f, f, f, f, kw.get("S", S), kw.get("N", 4), kw.get("H", 2),
                                       kw.get("dk", 64), kw.get("dv", 64), kw.get("dt", E.KDA_BF16),
                                       kw.get("o", o), None)
    assert call(dk=96) == E.KDA_ERR_UNSUPPORTED
    assert call(N=-1) == E.KDA_ERR_INVALID_ARG
    assert call(N=0) == E.KDA_OK
    assert call(q=None) == E.KDA_ERR_INVALID_ARG
    assert call(o=f) == E.KDA_ERR_INVALID_ARG            # o aliases an input
    assert call(S=P(0x4004)) == E.KDA_ERR_INVALID_ARG    # state not 16-byte aligned
    assert call(dt=3) == E.KDA_ERR_INVALID_ARG


def test_verify_argument_checks(lib):
    """kda_decode_multi refuses before any launch: more tokens than the kernel
    stages (16), negative sizes, unsupported head dims, null or aliased
    pointers, an unaligned state; N = 0 or K = 0 is a no-op."""
    P = ctypes.c_void_p
    f = P(0x1000)
    S = P(0x4000)
    o = P(0x5000)
    E = _lib
    call = lambda **kw: lib.kda_decode_multi(kw.get("q", f), f, f, f, f, kw.get("S", S), None, kw.get("N", 4),
                                             kw.get("K", 4), kw.get("H", 2), kw.get("dk", 64), kw.get("dv", 64),
                                             kw.get("dt", E.KDA_BF16), kw.get("o", o), None)
    assert call(K=17) == E.KDA_ERR_UNSUPPORTED
    assert call(K=-1) == E.KDA_ERR_INVALID_ARG
    assert call(N=-1) == E.KDA_ERR_INVALID_ARG
    assert call(K=0) == E.KDA_OK
    assert call(N=0) == E.KDA_OK
    assert call(dk=96) == E.KDA_ERR_UNSUPPORTED
    assert call(q=None) == E.KDA_ERR_INVALID_ARG
    assert call(o=f) == E.KDA_ERR_INVALID_ARG            # o aliases an input
    assert call(S=P(0x4004)) == E.KDA_ERR_INVALID_ARG    # state not 16-byte aligned
    assert call(dt=3) == E.KDA_ERR_INVALID_ARG


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(ImportError):
        _lib.load()
