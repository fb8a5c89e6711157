"""Failure detection on the device without a GPU fault.

Every wait inside the library's kernels is bounded in time.  The self-test
kernel waits on an mbarrier phase that nothing completes, with a 2 ms limit:
the wait must give up, record the timeout in the device status word and let
the kernel return, so that fa_last_device_error reports it, clears it, and
the context stays usable for real work.
"""
import ctypes
import time

import pytest
import torch

import exact_attention_39_gb300 as fa
from exact_attention_39_gb300 import binding as b
from exact_attention_39_gb300 import workloads as W


@pytest.mark.gpu
def test_bounded_wait_reports_timeout_and_context_survives():
    assert fa.last_device_error() == b.FA_OK          # clean before
    t0 = time.perf_counter()
    assert b.selftest_wait_timeout(2_000_000) == b.FA_OK
    assert fa.last_device_error() == b.FA_ERR_DEVICE_TIMEOUT
    assert time.perf_counter() - t0 < 10.0
    assert fa.last_device_error() == b.FA_OK          # read once, then cleared
    # the GPU still computes correctly afterwards
    w = W.TINY
    q, k, v = (t.cuda() for t in W.make_inputs(w))
    o1, _ = fa.fwd(q, k, v, scale=w.scale)
    o2, _ = fa.fwd(q, k, v, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.last_device_error() == b.FA_OK
    assert torch.equal(o1, o2) and torch.isfinite(o1.float()).all()


def test_selftest_limits_checked_on_host():
    lib = b.load_library()
    assert lib.fa_selftest_wait_timeout(10, ctypes.c_void_p(0)) == b.FA_ERR_SHAPE
    assert lib.fa_selftest_wait_timeout(5_000_000_000, ctypes.c_void_p(0)) == b.FA_ERR_SHAPE
