"""fa_bwd_noalloc: the backward for callers that cannot allocate device
memory (a plug-in inside a host program that owns every allocation, or a
loop that may not pay for one).  It keeps its row-sum scratch in the
library's static device memory instead of a caller workspace.

This file is collected last on purpose.  The GPU test calls the entry point
through the C ABI twice in a row, on different problems, and checks each
result against fa_bwd with a workspace: the two run the same kernels on the
same inputs, so they must agree exactly -- inside every tolerance the parity
tests use.  It passes alone in a fresh process (the first call sets up the
scratch address) and after the other tests.
"""
import ctypes

import pytest
import torch

import exact_attention_39_gb300 as fa
from exact_attention_39_gb300 import binding as b
from exact_attention_39_gb300 import workloads as W


def _inputs(w):
    dev = torch.device("cuda")
    q, k, v = (t.to(dev) for t in W.make_inputs(w))
    g = W.make_upstream_grad(w).to(dev)
    o, lse = fa.fwd(q, k, v, causal=w.causal, scale=w.scale)
    return q, k, v, o, lse, g


def _noalloc(q, k, v, o, lse, g, w):
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    code = b.FA_BF16 if w.dtype == "bf16" else b.FA_FP16
    st = b.fa_bwd_noalloc_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                              g.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                              dv.data_ptr(), w.B, w.H, w.N, w.d, w.causal, w.scale, code,
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == b.FA_OK, b.status_string(st)
    return dq, dk, dv


@pytest.mark.gpu
def test_noalloc_backward_matches_workspace_backward_twice():
    cases = [W.Workload("na1", 2, 4, 700, 64, "bf16", True, seed=21),
             W.Workload("na2", 1, 3, 300, 128, "fp16", False, seed=22)]
    for w in cases:                       # two calls in a row, different problems
        args = _inputs(w)
        got = _noalloc(*args, w)
        torch.cuda.synchronize()
        assert fa.last_device_error() == 0
        ref = fa.bwd(*args[:5], args[5], causal=w.causal, scale=w.scale)
        torch.cuda.synchronize()
        for a, r, name in zip(got, ref, ("dq", "dk", "dv")):
            assert torch.isfinite(a.float()).all(), name
            assert torch.equal(a, r), (w.name, name, (a.float() - r.float()).abs().max().item())


def test_noalloc_rejects_problems_beyond_its_scratch():
    # B * H * N over the static capacity: FA_ERR_WORKSPACE before any CUDA call
    P = 0x10000
    n_over = b.FA_BWD_NOALLOC_MAX_ROWS // 32 + 128
    st = b.fa_bwd_noalloc_raw(P, P, P, P, P, P, P, P, P, 1, 32, n_over, 64, 0, 0.125,
                              b.FA_BF16, ctypes.c_void_p(0))
    assert st == b.FA_ERR_WORKSPACE
    assert b.fa_bwd_noalloc_raw(0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 1, 1, 64, 0, 0.125,
                                b.FA_BF16, ctypes.c_void_p(0)) == b.FA_OK


def test_noalloc_checks_arguments_like_fa_bwd_before_any_cuda_call():
    # A problem of exactly the scratch's capacity passes the capacity check
    # and then meets fa_bwd's own checks, which run before anything touches
    # CUDA (so these hold on a machine without a GPU).
    P = 0x10000
    s0 = ctypes.c_void_p(0)
    cap = b.FA_BWD_NOALLOC_MAX_ROWS
    n_at_cap = cap // 32                  # B = 1, H = 32: exactly the capacity
    assert n_at_cap % 128 == 0
    assert b.fa_bwd_noalloc_raw(0, 0, 0, 0, 0, 0, 0, 0, 0, 1, 32, n_at_cap, 64, 0, 0.125,
                                b.FA_BF16, s0) == b.FA_ERR_NULL
    # one padded block more is over the capacity
    assert b.fa_bwd_noalloc_raw(P, P, P, P, P, P, P, P, P, 1, 32, n_at_cap + 1, 64, 0,
                                0.125, b.FA_BF16, s0) == b.FA_ERR_WORKSPACE
    # fa_bwd's errors, not a CUDA error, for bad arguments of an in-range shape
    assert b.fa_bwd_noalloc_raw(P, P, P, P, P, P, P, P, P, 1, 2, 256, 96, 0, 0.125,
                                b.FA_BF16, s0) == b.FA_ERR_HEADDIM
    assert b.fa_bwd_noalloc_raw(P, P, P, P, P, P, P, P, P, 1, 2, 256, 64, 0, 0.125,
                                7, s0) == b.FA_ERR_DTYPE
    assert b.fa_bwd_noalloc_raw(P, P, P, P, P, P, P, P, P, 1, 2, 256, 64, 0, -1.0,
                                b.FA_BF16, s0) == b.FA_ERR_SCALE
    assert b.fa_bwd_noalloc_raw(P, P, P, P, P, P, P + 8, P, P, 1, 2, 256, 64, 0, 0.125,
                                b.FA_BF16, s0) == b.FA_ERR_ALIGN


def test_noalloc_and_bwd_reject_shapes_that_overflow():
    # B * H beyond 2^31 - 1, and N whose padding to whole blocks leaves int
    P = 0x10000
    s0 = ctypes.c_void_p(0)
    big = 1 << 16
    assert b.fa_bwd_noalloc_raw(P, P, P, P, P, P, P, P, P, big, big, 1 << 30, 64, 0, 0.125,
                                b.FA_BF16, s0) == b.FA_ERR_SHAPE
    assert b.fa_bwd_raw(P, P, P, P, P, P, P, P, P, P, 1 << 40, big, big, 1 << 30, 64, 0,
                        0.125, b.FA_BF16, s0) == b.FA_ERR_SHAPE
    n_max = (1 << 31) - 1
    assert b.fa_bwd_noalloc_raw(P, P, P, P, P, P, P, P, P, 1, 1, n_max, 64, 0, 0.125,
                                b.FA_BF16, s0) == b.FA_ERR_SHAPE
    assert b.fa_bwd_raw(P, P, P, P, P, P, P, P, P, P, 1 << 40, 1, 1, n_max, 64, 0, 0.125,
                        b.FA_BF16, s0) == b.FA_ERR_SHAPE


def test_binding_capacity_matches_the_header():
    # the binding's copy of the scratch capacity is the header's #define
    import os
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    with open(os.path.join(root, "include", "fa.h")) as f:
        m = re.search(r"#define\s+FA_BWD_NOALLOC_MAX_ROWS\s+\(1LL\s*<<\s*(\d+)\)", f.read())
    assert m, "FA_BWD_NOALLOC_MAX_ROWS not found in include/fa.h"
    assert b.FA_BWD_NOALLOC_MAX_ROWS == 1 << int(m.group(1))
