"""Exact attention forward for GB300 (sm_103a).

``fwd(q, k, v, causal, scale)`` computes O = softmax(scale * Q K^T [+ causal
mask]) V and the per-row logsumexp with the hand-written tcgen05 kernel in
``csrc/`` through the C ABI of ``include/fa.h``.  The shared library is
loaded on first use; without it every call raises (no CPU fallback).
"""
from .binding import (FaError, bwd, bwd_workspace_bytes, fwd,  # noqa: F401
                      fwd_fp8, fwd_host, last_device_error, load_library,
                      status_string, version)
from . import workloads  # noqa: F401
from .shard import fwd_shard, head_range  # noqa: F401

__all__ = ["fwd", "fwd_fp8", "fwd_host", "bwd", "bwd_workspace_bytes", "last_device_error", "load_library",
           "status_string", "version", "FaError", "workloads", "fwd_shard", "head_range"]
