"""The fp64 CPU oracle for KDA.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline legs of ``bench.py`` may import this package.  The CUDA library
never calls it, links it or falls back to it, and it shares no code with it.

* ``prefill``   -- the per-token recurrence in C (``kda_ref.c``), fp64,
  OpenMP over (sequence, head).  This is the oracle every GPU result is
  compared with.  Decode is the same call with one token per sequence.
* ``prefill_fused`` / ``decode_fused`` / ``prologue`` -- the same recurrence
  behind the parameter-free prologue of the Kimi Linear layer (q, k
  L2-normalised, log-decay = clamp(-softplus(gate), -5, -1e-4), beta =
  sigmoid(beta_logit)), also in ``kda_ref.c``.
* ``chunked``   -- the pages' FlashKDA chunk form in fp64 numpy, used only to
  cross-check the token loop (pin P5).

Every function cites the passage it follows in its own docstring/comment.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_ref.c")
_LIB_PATH = os.path.join(_HERE, "libkda_ref.so")
_lock = threading.Lock()
_lib = None


def compile_source(src: str, out: str) -> str:
    """gcc -O2 -fopenmp: one C file to one shared library."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``kda_ref.c`` into ``oracle/libkda_ref.so`` (gcc, OpenMP)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


def bind(path: str):
    """Open a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    lib.kda_ref_prefill.argtypes = [P, P, P, P, P, P, P, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    P, P, ctypes.c_int]
    lib.kda_ref_prefill.restype = ctypes.c_int
    lib.kda_ref_prefill_prologue.argtypes = lib.kda_ref_prefill.argtypes
    lib.kda_ref_prefill_prologue.restype = ctypes.c_int
    I = ctypes.c_int
    lib.kda_ref_prologue.argtypes = [P, I, I, P, P, I, P, P, I, P]
    lib.kda_ref_prologue.restype = None
    lib.kda_ref_max_threads.argtypes = []
    lib.kda_ref_max_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind(build())
    return _lib


def max_threads() -> int:
    return int(_load().kda_ref_max_threads())


def _f32(x):
    if hasattr(x, "detach"):  # a torch tensor: widen the stored values exactly
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float32).numpy()
    return np.ascontiguousarray(x, dtype=np.float32)


def prefill(q, k, v, log_alpha, beta, cu_seqlens=None, S0=None, heads=None,
            n_threads: int = 0, want_O: bool = True, lib=None, _prologue: bool = False):
    """Per-token fp64 KDA over a packed varlen batch (the definition).

    q, k, log_alpha: [T, H, dk]; v: [T, H, dv]; beta: [T, H] (numpy or torch,
    any float dtype -- values are widened exactly to fp32 then fp64);
    cu_seqlens: [n_seq+1] (None = one sequence of T tokens);
    S0: [n_seq, H, dk, dv] or None (zeros); heads: (h0, h1) or None (all).
    ``lib`` (tests only) runs another build of the same C source.
    Returns (O [T, Hs, dv] or None, S_final [n_seq, Hs, dk, dv]) as fp64.
    """
    lib = lib or _load()
    q, k, v, log_alpha, beta = (_f32(x) for x in (q, k, v, log_alpha, beta))
    T, H, dk = q.shape
    dv = v.shape[2]
    if cu_seqlens is None:
        cu = np.array([0, T], dtype=np.int64)
    else:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens),
                                  dtype=np.int64)
    n_seq = len(cu) - 1
    h0, h1 = (0, H) if heads is None else heads
    Hs = h1 - h0
    s0 = None
    if S0 is not None:
        if hasattr(S0, "detach"):
            import torch
            S0 = S0.detach().to("cpu").to(torch.float64).numpy()
        s0 = np.ascontiguousarray(S0, dtype=np.float64)
        assert s0.shape == (n_seq, H, dk, dv)
    O = np.empty((T, Hs, dv), dtype=np.float64) if want_O else None
    Sf = np.empty((n_seq, Hs, dk, dv), dtype=np.float64)
    ptr = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    fn = lib.kda_ref_prefill_prologue if _prologue else lib.kda_ref_prefill
    rc = fn(ptr(q), ptr(k), ptr(v), ptr(log_alpha), ptr(beta), ptr(s0), ptr(cu),
            n_seq, H, dk, dv, h0, h1, ptr(O), ptr(Sf), int(n_threads))
    if rc != 0:
        raise ValueError(f"kda_ref_prefill failed with code {rc}")
    return O, Sf


def prefill_fused(q, k, v, gate, beta_logit, cu_seqlens=None, S0=None, heads=None, n_threads: int = 0,
                  want_O: bool = True):
    """``prefill`` behind the parameter-free prologue: q, k unnormalised,
    gate [T, H, dk] and beta_logit [T, H] the pre-activations of log_alpha and
    beta ("Kimi K3: the manos, the mythos, the legendos", section "Kimi Linear";
    "LLM architecture at trillion scale", section "The KDA update, in plain
    words")."""
    return prefill(q, k, v, gate, beta_logit, cu_seqlens=cu_seqlens, S0=S0, heads=heads, n_threads=n_threads,
                   want_O=want_O, _prologue=True)


def decode_fused(q, k, v, gate, beta_logit, S, n_threads: int = 0):
    """``decode`` behind the parameter-free prologue (see ``prefill_fused``)."""
    N = q.shape[0]
    cu = np.arange(N + 1, dtype=np.int64)
    return prefill_fused(q, k, v, gate, beta_logit, cu_seqlens=cu, S0=S, n_threads=n_threads)


def prologue(x=None, gate=None, beta_logit=None):
    """The prologue alone, fp64: x [..., d] -> x / sqrt(sum x^2 + 1e-6) over the
    last axis; gate -> clamp(-softplus(gate), -5, -1e-4); beta_logit ->
    sigmoid(beta_logit).  Returns (x_hat, log_alpha, beta), None where no input."""
    lib = _load()
    ptr = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    xh = la = bt = None
    xf = gf = bf = None
    n_rows = d = n_g = n_b = 0
    if x is not None:
        xf = _f32(x)
        d = xf.shape[-1]
        n_rows = xf.size // d
        xh = np.empty(xf.shape, dtype=np.float64)
    if gate is not None:
        gf = _f32(gate)
        n_g = gf.size
        la = np.empty(gf.shape, dtype=np.float64)
    if beta_logit is not None:
        bf = _f32(beta_logit)
        n_b = bf.size
        bt = np.empty(bf.shape, dtype=np.float64)
    lib.kda_ref_prologue(ptr(xf), n_rows, d, ptr(xh), ptr(gf), n_g, ptr(la), ptr(bf), n_b, ptr(bt))
    return xh, la, bt


def decode(q, k, v, log_alpha, beta, S, n_threads: int = 0):
    """One decode step = the recurrence for a single token per sequence.

    q, k, log_alpha: [N, H, dk]; v: [N, H, dv]; beta: [N, H]; S: [N, H, dk, dv].
    Returns (o [N, H, dv], S_new [N, H, dk, dv]) as fp64.
    """
    N = q.shape[0]
    cu = np.arange(N + 1, dtype=np.int64)
    return prefill(q, k, v, log_alpha, beta, cu_seqlens=cu, S0=S, n_threads=n_threads)


from . import chunked  # noqa: E402  (re-export)
