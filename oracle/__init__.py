"""fp64 CPU oracle for the exact attention forward.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg import this package; the product path
(``exact_attention_39_gb300``) never does, and the two share no code.

``attention_fwd`` follows the plain definition of attention: scale, mask,
softmax, weighted sum (zzycbzc.com/news/393333, section
"算子融合的极致优化", item 2), written out as a two-pass row computation in
``attn_oracle.c``.  ``brute.attention_brute`` is an unfused pure-Python
restatement used to cross-check it on tiny shapes.

Pins (tests/test_oracle.py): hand-derived worked examples in
tests/golden/, closed forms (Q = 0, constant V, one key, causal first row),
invariants (key/value permutation, per-row logit shift, scale folding),
and agreement with the brute force.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force=False):
    """Compile liboracle.so with gcc (plain C, -O2, no fast-math)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-fno-fast-math", "-std=c11", "-fPIC", "-shared",
           "-Wall", "-o", tmp, _SRC, "-lpthread", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        dp = ctypes.POINTER(ctypes.c_double)
        lp = ctypes.POINTER(ctypes.c_long)
        lib.fa_oracle_fwd.argtypes = [
            dp, dp, dp, ctypes.c_long, ctypes.c_long, ctypes.c_long,
            ctypes.c_long, ctypes.c_int, ctypes.c_double, lp, ctypes.c_long,
            dp, dp, ctypes.c_int]
        lib.fa_oracle_fwd.restype = ctypes.c_int
        lib.fa_oracle_row_weights.argtypes = [
            dp, dp, dp, ctypes.c_long, ctypes.c_long, ctypes.c_long,
            ctypes.c_int, ctypes.c_double, ctypes.c_long, dp]
        lib.fa_oracle_row_weights.restype = ctypes.c_long
        lib.fa_oracle_bwd.argtypes = [
            dp, dp, dp, dp, ctypes.c_long, ctypes.c_long, ctypes.c_long,
            ctypes.c_long, ctypes.c_int, ctypes.c_double, dp, dp, dp,
            ctypes.c_int]
        lib.fa_oracle_bwd.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(a):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    return a


def _dptr(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads():
    return os.cpu_count() or 1


def attention_fwd(q, k, v, scale, causal, rows=None, nthreads=None):
    """Exact attention forward in fp64.

    q: [..., Nq, d]; k, v: [..., Nk, d] (leading dims are independent
    problems, e.g. batch and heads).  ``rows`` optionally selects query
    rows (the same subset in every problem).

    Returns (O [..., R, d] float64, LSE [..., R] float64), R = Nq or
    len(rows).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    lead = q.shape[:-2]
    nq, d = q.shape[-2], q.shape[-1]
    nk = k.shape[-2]
    if k.shape[:-2] != lead or v.shape != k.shape or k.shape[-1] != d:
        raise ValueError("q, k, v shapes disagree")
    bh = int(np.prod(lead)) if lead else 1
    lib = _load()
    if rows is None:
        nrows = nq
        rows_arr = None
        rows_ptr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows_arr.size
        rows_ptr = rows_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_long))
    o = np.empty(lead + (nrows, d), dtype=np.float64)
    lse = np.empty(lead + (nrows,), dtype=np.float64)
    nt = default_threads() if nthreads is None else int(nthreads)
    rc = lib.fa_oracle_fwd(_dptr(q), _dptr(k), _dptr(v), bh, nq, nk, d,
                           int(bool(causal)), float(scale), rows_ptr, nrows,
                           _dptr(o), _dptr(lse), nt)
    if rc != 0:
        raise ValueError("fa_oracle_fwd rejected its arguments")
    return o, lse


def attention_bwd(q, k, v, dout, scale, causal, nthreads=None):
    """Gradients (dQ, dK, dV) of L = sum(O * dout) for O = attention(q, k, v),
    in fp64, shapes as attention_fwd (dout like q)."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    lead = q.shape[:-2]
    nq, d = q.shape[-2], q.shape[-1]
    nk = k.shape[-2]
    if (k.shape[:-2] != lead or v.shape != k.shape or k.shape[-1] != d
            or dout.shape != q.shape):
        raise ValueError("q, k, v, dout shapes disagree")
    bh = int(np.prod(lead)) if lead else 1
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    nt = default_threads() if nthreads is None else int(nthreads)
    rc = _load().fa_oracle_bwd(_dptr(q), _dptr(k), _dptr(v), _dptr(dout), bh,
                               nq, nk, d, int(bool(causal)), float(scale),
                               _dptr(dq), _dptr(dk), _dptr(dv), nt)
    if rc != 0:
        raise ValueError("fa_oracle_bwd rejected its arguments")
    return dq, dk, dv


def row_weights(q, k, v, scale, causal, i):
    """Normalised softmax weights of query row ``i`` of one head ([Nk])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    nq, d = q.shape
    nk = k.shape[0]
    p = np.empty(nk, dtype=np.float64)
    n = _load().fa_oracle_row_weights(_dptr(q), _dptr(k), _dptr(v), nq, nk,
                                      d, int(bool(causal)), float(scale),
                                      int(i), _dptr(p))
    if n < 0:
        raise ValueError("fa_oracle_row_weights rejected its arguments")
    return p
