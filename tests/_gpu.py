"""Shared helpers for the GPU parity tests (compare the CUDA path with the oracle)."""
import numpy as np
import pytest
import torch

TOL_FP32 = 1e-4      # max|gpu - ref| / max|ref| for fp32 inputs
TOL_BF16 = 5e-3      # ... for bf16 inputs (fp32 state)


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from kimi_delta_attention_chunked_gb300 import build
    build.build()
    return torch.device("cuda", 0)


def rel_err(gpu, ref):
    g = gpu.detach().double().cpu().numpy() if hasattr(gpu, "detach") else np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), "non-finite GPU output"
    denom = max(float(np.max(np.abs(r))), 1e-30)
    return float(np.max(np.abs(g - r))) / denom


def tol_for(dtype):
    return TOL_BF16 if dtype == torch.bfloat16 else TOL_FP32
