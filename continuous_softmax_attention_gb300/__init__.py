"""GB300-native forward pass of causal Continuous Softmax Attention.

The compute lives in ``libcsa.so`` (hand-written CUDA for sm_103a behind a
C ABI, declared in ``include/csa.h``).  This package is the thin ctypes
binding over that library; nothing here computes attention.  Calls fail
loudly when the library has not been built.
"""
from .inputs import ZERO, COPY_FIRST, GIVEN  # noqa: F401
from ._lib import (  # noqa: F401
    CsaError,
    HostForwardPipeline,
    backward,
    backward_workspace_bytes,
    decode,
    decode_merge_ranges,
    decode_noalloc,
    decode_range,
    decode_range_workspace_bytes,
    decode_workspace_bytes,
    device_status,
    forward,
    forward_host,
    forward_host_workspace_bytes,
    forward_symmetric,
    logphi2_eval,
    segment_weights_eval,
    selftest_forward_delay,
    selftest_wait_timeout,
    shard_rows,
    status_string,
    std_forward,
)

__all__ = [
    "ZERO", "COPY_FIRST", "GIVEN", "CsaError", "forward", "forward_host", "HostForwardPipeline",
    "forward_host_workspace_bytes", "forward_symmetric", "std_forward",
    "backward",
    "backward_workspace_bytes", "decode", "decode_noalloc", "decode_workspace_bytes",
    "decode_range", "decode_range_workspace_bytes", "decode_merge_ranges", "shard_rows",
    "logphi2_eval",
    "segment_weights_eval", "device_status", "selftest_forward_delay", "selftest_wait_timeout",
    "status_string",
]
