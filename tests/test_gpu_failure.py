"""Failure detection on the GPU, without a GPU fault: a kernel that waits on an
mbarrier nothing completes gives up after its bounded wait, records
KDA_ERR_TIMEOUT in the device status word, and returns; the host reads the
word, and the next calls run normally."""
import pytest
import torch

import oracle
import kimi_delta_attention_chunked_gb300 as kda
from kimi_delta_attention_chunked_gb300 import _lib, inputs
from _gpu import need_gpu, rel_err

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_the_device_stays_usable():
    dev = need_gpu()
    kda.kda_get_last_device_status()                       # start from a clear word
    kda.kda_check_wait_timeout(20_000_000)                 # ~10 ms of SM clock
    assert kda.kda_get_last_device_status() == _lib.KDA_ERR_TIMEOUT
    assert kda.kda_get_last_device_status() == _lib.KDA_OK  # reading clears it
    # the context still works: a decode step against the oracle
    w = inputs.Workload("after_timeout", "decode", H=2, dk=128, dv=128, dtype=torch.bfloat16, B=4, s0_std=0.02)
    d = inputs.make_decode(w, device=dev, seed=1)
    S = d["S"].clone()
    o = kda.kda_decode(d["q"][0], d["k"][0], d["v"][0], d["log_alpha"][0], d["beta"][0], S)
    torch.cuda.synchronize()
    assert kda.kda_get_last_device_status() == _lib.KDA_OK
    o_ref, S_ref = oracle.decode(d["q"][0], d["k"][0], d["v"][0], d["log_alpha"][0], d["beta"][0], d["S"])
    assert rel_err(o, o_ref) <= 5e-3
    assert rel_err(S, S_ref) <= 5e-3
