"""kda_prefill_noalloc: the prefill entry point for callers that cannot
allocate device memory (their runtime owns all device memory, or their plugin
interface hands the library only inputs and outputs).  It uses a fixed device
array inside the library as its workspace.

Checked here through the C ABI: its outputs equal those of kda_prefill with a
caller-allocated workspace, on two calls in a row (the array keeps the first
call's contents, which must not leak into the second), and a problem too big
for the array is refused before anything runs.  This file is collected last
so that a failure here cannot hide another test's result."""
import pytest
import torch

import kimi_delta_attention_chunked_gb300 as kda
from kimi_delta_attention_chunked_gb300 import _lib, inputs
from _gpu import need_gpu, rel_err

pytestmark = pytest.mark.gpu

TOL = 5e-3


def _case(dev, lengths, seed):
    w = inputs.Workload("noalloc", "prefill", H=4, dk=128, dv=128, dtype=torch.bfloat16, chunk=64, s0_std=0.02)
    return inputs.make_prefill(w, device=dev, seed=seed, lengths=lengths)


def _both(d):
    args = (d["q"], d["k"], d["v"], d["log_alpha"], d["beta"])
    kw = dict(S0=d["S0"], cu_seqlens=d["cu_seqlens"], cu_seqlens_host=d["cu_seqlens_host"], chunk=64)
    O_ref, S_ref = kda.kda_prefill(*args, **kw)
    O = torch.full_like(O_ref, float("nan"))
    S = torch.full_like(S_ref, float("nan"))
    kda.kda_prefill_noalloc(*args, O=O, S_final=S, **kw)
    torch.cuda.synchronize()
    assert kda.kda_get_last_device_status() == 0
    return (O, S), (O_ref.double().cpu().numpy(), S_ref.double().cpu().numpy())


def test_noalloc_matches_prefill_on_two_calls():
    dev = need_gpu()
    # two different problems back to back: the second must not see the first's scratch
    for lengths, seed in (([300, 77, 1], 21), ([64, 5, 129], 22)):
        (O, S), (O_ref, S_ref) = _both(_case(dev, lengths, seed))
        assert rel_err(O, O_ref) <= TOL
        assert rel_err(S, S_ref) <= TOL


def test_noalloc_rejects_problems_larger_than_its_array():
    dev = need_gpu()
    lib = _lib.load()
    T, H = 1 << 16, 32
    need = kda.kda_prefill_workspace_size(1, T, H, 128, 128, 64, torch.bfloat16)
    assert need > _lib.NOALLOC_SCRATCH_BYTES
    fake = torch.empty(16, dtype=torch.uint8, device=dev)
    p = fake.data_ptr()
    st = lib.kda_prefill_noalloc(p, p, p, p, p, None, None, None, 1, T, H, 128, 128, 64, _lib.KDA_BF16,
                                 p + 4096, None, None)
    assert st == _lib.KDA_ERR_WORKSPACE
