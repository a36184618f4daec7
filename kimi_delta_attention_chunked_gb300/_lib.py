"""ctypes binding of ``libkda.so`` -- argument marshalling only.

Every function here has the name of the C entry point it calls (see
``include/kda.h``).  Tensors are passed as raw device pointers; PyTorch is used
only to allocate outputs and workspaces and to name the current stream.  There
is no fallback: if the library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkda.so")
LIB_DEBUG_PATH = os.path.join(_PKG, "libkda_debug.so")

(KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_WORKSPACE, KDA_ERR_CUDA, KDA_ERR_TIMEOUT,
 KDA_ERR_PRECONDITION, KDA_ERR_DEVICE_CHECK) = range(8)
KDA_FP32, KDA_BF16 = 0, 1
SYMBOLS = ("kda_prefill_workspace_size", "kda_prefill", "kda_prefill_ckpt", "kda_prefill_fused",
           "kda_prefill_noalloc", "kda_decode", "kda_decode_fused", "kda_decode_multi",
           "kda_get_last_device_status", "kda_check_wait_timeout", "kda_set_trace_events", "kda_debug_build",
           "kda_status_string")
NOALLOC_SCRATCH_BYTES = 64 << 20

_lock = threading.Lock()
_lib = None
_lib_debug = None


class KDAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {kda_status_string(status)}")


def load():
    """Load libkda.so (built by ``build.build()``); raises if it is not there."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = _open(LIB_PATH)
        return _lib


def load_debug():
    """Load libkda_debug.so, the variant with the input precondition and device
    index checks (include/kda.h, kda_debug_build); raises if it is not there.
    The functions of this module call the release library; the debug one is
    called through the returned ctypes handle."""
    global _lib_debug
    with _lock:
        if _lib_debug is None:
            _lib_debug = _open(LIB_DEBUG_PATH)
        return _lib_debug


def _open(path):
    if not os.path.exists(path):
        raise ImportError(f"KDA CUDA library not built: {path} is missing "
                          "(run python -m kimi_delta_attention_chunked_gb300.build)")
    lib = ctypes.CDLL(path)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.kda_prefill_workspace_size.argtypes = [I, I, I, I, I, I, I]
    lib.kda_prefill_workspace_size.restype = Z
    lib.kda_prefill.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, P, P, Z, P]
    lib.kda_prefill.restype = I
    lib.kda_prefill_ckpt.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, P, I, P, I, P, Z, P]
    lib.kda_prefill_ckpt.restype = I
    lib.kda_prefill_fused.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, P, P, Z, P]
    lib.kda_prefill_fused.restype = I
    lib.kda_decode_fused.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, P]
    lib.kda_decode_fused.restype = I
    lib.kda_prefill_noalloc.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, P, P]
    lib.kda_prefill_noalloc.restype = I
    lib.kda_decode.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, P]
    lib.kda_decode.restype = I
    lib.kda_decode_multi.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, P, P]
    lib.kda_decode_multi.restype = I
    lib.kda_get_last_device_status.argtypes = [P]
    lib.kda_get_last_device_status.restype = I
    lib.kda_check_wait_timeout.argtypes = [ctypes.c_longlong, P]
    lib.kda_check_wait_timeout.restype = I
    lib.kda_set_trace_events.argtypes = [P, I]
    lib.kda_set_trace_events.restype = I
    lib.kda_debug_build.argtypes = []
    lib.kda_debug_build.restype = I
    lib.kda_status_string.argtypes = [I]
    lib.kda_status_string.restype = ctypes.c_char_p
    return lib


def kda_status_string(status: int) -> str:
    return load().kda_status_string(int(status)).decode()


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.bfloat16:
        return KDA_BF16
    if t == torch.float32:
        return KDA_FP32
    raise TypeError(f"KDA supports bfloat16 and float32 q/k/v, not {t}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _on(device, fn, *args):
    """Call a C entry point with ``device`` current: the library picks the SM
    count, its internal stream and the no-workspace array from the current
    device, which must be the one that holds the tensors."""
    with torch.cuda.device(device):
        return fn(*args)


def _check_dev(name, t, device, dtype=None):
    if t is None:
        return
    if not t.is_cuda or t.device != device:
        raise ValueError(f"{name} must be on {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _check_shape(name, t, shape):
    """The kernels index every tensor from the sizes passed through the C ABI
    (which sees only pointers), so a tensor of another shape would be read or
    written out of bounds: refuse it here."""
    if t is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _token_shapes(q, v, lead):
    """(dk, dv) of q [*lead, dk] and v [*lead, dv], checking their leading dims."""
    if q.dim() != len(lead) + 1 or v.dim() != len(lead) + 1:
        raise ValueError(f"q and v must have {len(lead) + 1} dims, got {q.dim()} and {v.dim()}")
    if tuple(v.shape[:-1]) != tuple(q.shape[:-1]):
        raise ValueError(f"v {tuple(v.shape)} does not match q {tuple(q.shape)} in its leading dims")
    return q.shape[-1], v.shape[-1]


def _check_prefill_shapes(q, k, v, log_alpha, beta, S0, cu_seqlens, cu_seqlens_host, O, S_final):
    """Shapes of a prefill call (include/kda.h): q, k, log_alpha [T, H, dk];
    v, O [T, H, dv]; beta [T, H]; S0, S_final [n_seq, H, dk, dv];
    cu_seqlens [n_seq + 1] (and its host copy).  Returns (T, H, dk, dv, n_seq)."""
    dk, dv = _token_shapes(q, v, ("T", "H"))
    T, H = q.shape[0], q.shape[1]
    _check_shape("k", k, (T, H, dk))
    _check_shape("log_alpha", log_alpha, (T, H, dk))
    _check_shape("beta", beta, (T, H))
    if cu_seqlens is not None and (cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1):
        raise ValueError("cu_seqlens must be a 1-D tensor of n_seq + 1 offsets")
    n_seq = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    if cu_seqlens is not None and cu_seqlens_host is not None and len(cu_seqlens_host) != n_seq + 1:
        raise ValueError(f"cu_seqlens_host must hold {n_seq + 1} offsets, got {len(cu_seqlens_host)}")
    _check_shape("S0", S0, (n_seq, H, dk, dv))
    _check_shape("O", O, (T, H, dv))
    _check_shape("S_final", S_final, (n_seq, H, dk, dv))
    return T, H, dk, dv, n_seq


def kda_prefill_workspace_size(n_seq: int, T_total: int, H: int, dk: int, dv: int, chunk: int,
                               dtype: torch.dtype) -> int:
    return int(load().kda_prefill_workspace_size(n_seq, T_total, H, dk, dv, chunk, _dtype_code(dtype)))


def kda_prefill(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None, cu_seqlens_host=None, chunk=64,
                O=None, S_final=None, workspace=None, stream=None, want_state=True):
    """Chunked prefill; returns (O, S_final).  Shapes as in ``include/kda.h``:
    q, k, log_alpha [T, H, dk]; v [T, H, dv]; beta [T, H]; S0 [n_seq, H, dk, dv] fp32 or
    None; cu_seqlens int32 [n_seq+1] on the device or None (one sequence)."""
    return _prefill("kda_prefill", q, k, v, log_alpha, beta, S0, cu_seqlens, cu_seqlens_host, chunk, O,
                    S_final, workspace, stream, want_state)


def kda_prefill_fused(q, k, v, gate, beta_logit, S0=None, cu_seqlens=None, cu_seqlens_host=None, chunk=64,
                      O=None, S_final=None, workspace=None, stream=None, want_state=True):
    """kda_prefill with the parameter-free prologue fused in (include/kda.h):
    q, k not normalised, gate and beta_logit are the pre-activations of
    log_alpha and beta.  Returns (O, S_final)."""
    return _prefill("kda_prefill_fused", q, k, v, gate, beta_logit, S0, cu_seqlens, cu_seqlens_host, chunk, O,
                    S_final, workspace, stream, want_state)


def _prefill(entry, q, k, v, log_alpha, beta, S0, cu_seqlens, cu_seqlens_host, chunk, O, S_final, workspace,
             stream, want_state):
    lib = load()
    dev = q.device
    T, H, dk, dv, n_seq = _check_prefill_shapes(q, k, v, log_alpha, beta, S0, cu_seqlens, cu_seqlens_host, O,
                                                S_final)
    for name, t in (("q", q), ("k", k), ("v", v), ("O", O)):
        _check_dev(name, t, dev, q.dtype)
    _check_dev("log_alpha", log_alpha, dev, torch.float32)
    _check_dev("beta", beta, dev, torch.float32)
    _check_dev("cu_seqlens", cu_seqlens, dev, torch.int32)
    _check_dev("S0", S0, dev, torch.float32)
    _check_dev("S_final", S_final, dev, torch.float32)
    if O is None:
        O = torch.empty((T, H, dv), dtype=q.dtype, device=dev)
    if S_final is None and want_state:
        S_final = torch.empty((n_seq, H, dk, dv), dtype=torch.float32, device=dev)
    host = None
    if cu_seqlens_host is not None:
        host = (ctypes.c_int32 * len(cu_seqlens_host))(*[int(x) for x in cu_seqlens_host])
    dt = _dtype_code(q.dtype)
    need = int(lib.kda_prefill_workspace_size(n_seq, T, H, dk, dv, chunk, dt))
    _check_dev("workspace", workspace, dev)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _on(dev, getattr(lib, entry), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(S0),
             _ptr(cu_seqlens), host, n_seq, T, H, dk, dv, chunk, dt, _ptr(O), _ptr(S_final),
             _ptr(workspace), ws_bytes, _stream(stream, dev))
    if st != KDA_OK:
        raise KDAError(st, entry)
    return O, S_final


def checkpoint_count(seq_lens, ckpt_every: int) -> int:
    """Number of checkpoints kda_prefill_ckpt writes for these sequence lengths."""
    return sum(int(n) // ckpt_every for n in seq_lens)


def kda_prefill_ckpt(q, k, v, log_alpha, beta, ckpt_every, S0=None, cu_seqlens=None, cu_seqlens_host=None,
                     chunk=64, O=None, S_final=None, ckpt=None, workspace=None, stream=None):
    """kda_prefill that also returns the state after every ``ckpt_every`` tokens
    of each sequence: (O, S_final, ckpt), ckpt [n_ckpt, H, dk, dv] fp32 with the
    checkpoints of sequence 0 first, in position order.  Without a ``ckpt``
    buffer the lengths must be known here (``cu_seqlens_host``, or one sequence)."""
    lib = load()
    dev = q.device
    T, H, dk, dv, n_seq = _check_prefill_shapes(q, k, v, log_alpha, beta, S0, cu_seqlens, cu_seqlens_host, O,
                                                S_final)
    if ckpt is not None and (ckpt.dim() != 4 or tuple(ckpt.shape[1:]) != (H, dk, dv)):
        raise ValueError(f"ckpt must have shape (n, {H}, {dk}, {dv}), got {tuple(ckpt.shape)}")
    for name, t in (("q", q), ("k", k), ("v", v), ("O", O)):
        _check_dev(name, t, dev, q.dtype)
    _check_dev("log_alpha", log_alpha, dev, torch.float32)
    _check_dev("beta", beta, dev, torch.float32)
    _check_dev("cu_seqlens", cu_seqlens, dev, torch.int32)
    _check_dev("S0", S0, dev, torch.float32)
    _check_dev("S_final", S_final, dev, torch.float32)
    if ckpt is None:
        if cu_seqlens is None:
            lens = [T]
        elif cu_seqlens_host is not None:
            b = [int(x) for x in cu_seqlens_host]
            lens = [b[i + 1] - b[i] for i in range(n_seq)]
        else:
            raise ValueError("kda_prefill_ckpt: pass ckpt or cu_seqlens_host")
        ckpt = torch.empty((checkpoint_count(lens, ckpt_every), H, dk, dv), dtype=torch.float32, device=dev)
    _check_dev("ckpt", ckpt, dev, torch.float32)
    if O is None:
        O = torch.empty((T, H, dv), dtype=q.dtype, device=dev)
    if S_final is None:
        S_final = torch.empty((n_seq, H, dk, dv), dtype=torch.float32, device=dev)
    host = None
    if cu_seqlens_host is not None:
        host = (ctypes.c_int32 * len(cu_seqlens_host))(*[int(x) for x in cu_seqlens_host])
    dt = _dtype_code(q.dtype)
    need = int(lib.kda_prefill_workspace_size(n_seq, T, H, dk, dv, chunk, dt))
    _check_dev("workspace", workspace, dev)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _on(dev, lib.kda_prefill_ckpt, _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(S0),
             _ptr(cu_seqlens), host, n_seq, T, H, dk, dv, chunk, dt, _ptr(O), _ptr(S_final),
             int(ckpt_every), _ptr(ckpt), ckpt.shape[0] if ckpt.numel() else 0,
             _ptr(workspace), ws_bytes, _stream(stream, dev))
    if st != KDA_OK:
        raise KDAError(st, "kda_prefill_ckpt")
    return O, S_final, ckpt


def kda_prefill_noalloc(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None, cu_seqlens_host=None, chunk=64,
                        O=None, S_final=None, stream=None):
    """kda_prefill with the library's fixed device scratch array as workspace,
    for callers that cannot allocate device memory (see include/kda.h).
    Outputs O and S_final must be passed in by such callers; allocating them
    here is only a convenience of this binding.  Returns (O, S_final)."""
    lib = load()
    dev = q.device
    T, H, dk, dv, n_seq = _check_prefill_shapes(q, k, v, log_alpha, beta, S0, cu_seqlens, cu_seqlens_host, O,
                                                S_final)
    for name, t in (("q", q), ("k", k), ("v", v), ("O", O)):
        _check_dev(name, t, dev, q.dtype)
    _check_dev("log_alpha", log_alpha, dev, torch.float32)
    _check_dev("beta", beta, dev, torch.float32)
    _check_dev("cu_seqlens", cu_seqlens, dev, torch.int32)
    _check_dev("S0", S0, dev, torch.float32)
    _check_dev("S_final", S_final, dev, torch.float32)
    if O is None:
        O = torch.empty((T, H, dv), dtype=q.dtype, device=dev)
    if S_final is None:
        S_final = torch.empty((n_seq, H, dk, dv), dtype=torch.float32, device=dev)
    host = None
    if cu_seqlens_host is not None:
        host = (ctypes.c_int32 * len(cu_seqlens_host))(*[int(x) for x in cu_seqlens_host])
    st = _on(dev, lib.kda_prefill_noalloc, _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(S0),
             _ptr(cu_seqlens), host, n_seq, T, H, dk, dv, chunk, _dtype_code(q.dtype),
             _ptr(O), _ptr(S_final), _stream(stream, dev))
    if st != KDA_OK:
        raise KDAError(st, "kda_prefill_noalloc")
    return O, S_final


def kda_decode(q, k, v, log_alpha, beta, S, o=None, stream=None):
    """One decode step; S [N, H, dk, dv] fp32 is updated in place; returns o [N, H, dv]."""
    return _decode("kda_decode", q, k, v, log_alpha, beta, S, o, stream)


def kda_decode_fused(q, k, v, gate, beta_logit, S, o=None, stream=None):
    """kda_decode with the parameter-free prologue fused in (see kda_prefill_fused)."""
    return _decode("kda_decode_fused", q, k, v, gate, beta_logit, S, o, stream)


def _decode(entry, q, k, v, log_alpha, beta, S, o, stream):
    lib = load()
    dev = q.device
    dk, dv = _token_shapes(q, v, ("N", "H"))
    N, H = q.shape[0], q.shape[1]
    _check_shape("k", k, (N, H, dk))
    _check_shape("log_alpha", log_alpha, (N, H, dk))
    _check_shape("beta", beta, (N, H))
    _check_shape("S", S, (N, H, dk, dv))
    _check_shape("o", o, (N, H, dv))
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        _check_dev(name, t, dev, q.dtype)
    _check_dev("log_alpha", log_alpha, dev, torch.float32)
    _check_dev("beta", beta, dev, torch.float32)
    _check_dev("S", S, dev, torch.float32)
    if o is None:
        o = torch.empty((N, H, dv), dtype=q.dtype, device=dev)
    st = _on(dev, getattr(lib, entry), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(S), N, H,
             dk, dv, _dtype_code(q.dtype), _ptr(o), _stream(stream, dev))
    if st != KDA_OK:
        raise KDAError(st, entry)
    return o


def kda_decode_multi(q, k, v, log_alpha, beta, S, commit_len=None, o=None, want_o=True, stream=None):
    """Verify K proposed tokens per sequence: q, k, log_alpha [N, K, H, dk]; v [N, K, H, dv];
    beta [N, K, H]; S [N, H, dk, dv] fp32 (written after commit_len[n] tokens; int32 [N] on
    the device or None = all K).  Returns o [N, K, H, dv] (None if want_o is False)."""
    lib = load()
    dev = q.device
    dk, dv = _token_shapes(q, v, ("N", "K", "H"))
    N, K, H = q.shape[0], q.shape[1], q.shape[2]
    _check_shape("k", k, (N, K, H, dk))
    _check_shape("log_alpha", log_alpha, (N, K, H, dk))
    _check_shape("beta", beta, (N, K, H))
    _check_shape("S", S, (N, H, dk, dv))
    _check_shape("commit_len", commit_len, (N,))
    _check_shape("o", o, (N, K, H, dv))
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        _check_dev(name, t, dev, q.dtype)
    _check_dev("log_alpha", log_alpha, dev, torch.float32)
    _check_dev("beta", beta, dev, torch.float32)
    _check_dev("S", S, dev, torch.float32)
    _check_dev("commit_len", commit_len, dev, torch.int32)
    if o is None and want_o:
        o = torch.empty((N, K, H, dv), dtype=q.dtype, device=dev)
    st = _on(dev, lib.kda_decode_multi, _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(S),
             _ptr(commit_len), N, K, H, dk, dv, _dtype_code(q.dtype), _ptr(o), _stream(stream, dev))
    if st != KDA_OK:
        raise KDAError(st, "kda_decode_multi")
    return o


_trace_keep = None


def kda_set_trace_events(events):
    """Record these torch.cuda.Event objects at the kernel boundaries of the
    following calls on this thread (None or [] stops)."""
    global _trace_keep
    lib = load()
    if not events:
        _trace_keep = None
        st = lib.kda_set_trace_events(None, 0)
    else:
        arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
        _trace_keep = (arr, list(events))
        st = lib.kda_set_trace_events(arr, len(events))
    if st != KDA_OK:
        raise KDAError(st, "kda_set_trace_events")


def kda_check_wait_timeout(limit_cycles: int, stream=None, device=None) -> None:
    """Runs one bounded wait that nothing completes (see include/kda.h); the
    next kda_get_last_device_status() then reports KDA_ERR_TIMEOUT."""
    dev = device or torch.device("cuda", torch.cuda.current_device())
    st = load().kda_check_wait_timeout(int(limit_cycles), _stream(stream, dev))
    if st != KDA_OK:
        raise KDAError(st, "kda_check_wait_timeout")


def kda_get_last_device_status(stream=None, device=None) -> int:
    dev = device or torch.device("cuda", torch.cuda.current_device())
    return int(load().kda_get_last_device_status(_stream(stream, dev)))
