"""Kimi Delta Attention (KDA) for one GB300 GPU.

The compute lives in ``libkda.so`` (hand-written sm_103a CUDA, C ABI declared
in ``include/kda.h``); this package only builds it and marshals arguments to
it.  ``inputs`` holds the seeded synthetic workloads.
"""
from ._lib import (KDAError, checkpoint_count, kda_check_wait_timeout, kda_decode, kda_decode_fused, kda_decode_multi,  # noqa: F401
                   kda_get_last_device_status, kda_prefill, kda_prefill_ckpt, kda_prefill_fused,
                   kda_prefill_noalloc, kda_prefill_workspace_size, kda_set_trace_events, kda_status_string, load)

__all__ = ["KDAError", "checkpoint_count", "kda_check_wait_timeout", "kda_decode", "kda_decode_fused", "kda_decode_multi",
           "kda_get_last_device_status", "kda_prefill", "kda_prefill_ckpt", "kda_prefill_fused",
           "kda_prefill_noalloc", "kda_prefill_workspace_size", "kda_set_trace_events", "kda_status_string",
           "load"]
