"""Chunked prefill for Kimi Delta Attention on GB300 (sm_103a).

The compute lives in hand-written CUDA kernels behind the C ABI of
include/kda.h (libkda_gb300.so, built in-tree by ``build.build()``); this
package is its thin Python binding.
"""
from ._binding import (  # noqa: F401
    PRE_GATE_LOGITS,
    PRE_NORM_QK,
    STATUS,
    STATUS_CODE,
    KdaError,
    check_device_error,
    chunk_prefill,
    chunk_prefill_backward,
    decode_step,
    kda_decode_step,
    kda_backward_workspace_bytes,
    kda_build_info,
    kda_chunk_prefill,
    kda_chunk_prefill_backward,
    kda_chunk_prefill_ex,
    kda_chunk_prefill_noalloc,
    kda_last_device_error,
    kda_set_backward_impl,
    kda_set_recurrent_impl,
    kda_set_scan_segments,
    kda_test_stall_recurrent,
    kda_stage_timing_begin,
    kda_stage_timing_end,
    kda_status_string,
    kda_workspace_bytes,
    kda_workspace_release,
    lib,
)

__version__ = "0.3.0"
