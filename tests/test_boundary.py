"""The C ABI boundary without a GPU: the library loads, exports every
symbol include/fa.h declares, and rejects bad arguments on the host before
touching CUDA."""
import ctypes
import os
import re

import pytest
import torch

import exact_attention_39_gb300 as fa
from exact_attention_39_gb300 import binding as b

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"FA_API\s+[\w\s\*]+?\b(fa_\w+)\s*\(", src)
    return names


def test_library_exports_every_declared_symbol():
    lib = fa.load_library()
    names = declared_symbols()
    assert "fa_fwd" in names and "fa_last_device_error" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(b.EXPORTED) <= set(names)


def test_version_and_status_strings():
    assert fa.version() >= 100
    for code in range(0, 9):
        s = fa.status_string(code)
        assert s and s != "unknown status"
    assert fa.status_string(99) == "unknown status"


P = 0x10000      # a 16-byte-aligned fake address: never dereferenced here
NULL = 0


def call(q=P, k=P, v=P, o=P, lse=P, B=1, H=1, N=128, d=64, causal=0,
         scale=0.125, dtype=b.FA_BF16):
    return b.fa_fwd_raw(q, k, v, o, lse, B, H, N, d, causal, scale, dtype,
                        ctypes.c_void_p(0))


@pytest.mark.parametrize("kw,code", [
    (dict(q=NULL), b.FA_ERR_NULL), (dict(k=NULL), b.FA_ERR_NULL),
    (dict(v=NULL), b.FA_ERR_NULL), (dict(o=NULL), b.FA_ERR_NULL),
    (dict(lse=NULL), b.FA_ERR_NULL),
    (dict(B=-1), b.FA_ERR_SHAPE), (dict(H=-2), b.FA_ERR_SHAPE),
    (dict(N=-1), b.FA_ERR_SHAPE), (dict(B=1 << 20, H=1 << 20), b.FA_ERR_SHAPE),
    (dict(d=32), b.FA_ERR_HEADDIM), (dict(d=96), b.FA_ERR_HEADDIM),
    (dict(d=0), b.FA_ERR_HEADDIM), (dict(dtype=2), b.FA_ERR_DTYPE),
    (dict(dtype=-1), b.FA_ERR_DTYPE),
    (dict(q=P + 8), b.FA_ERR_ALIGN), (dict(o=P + 2), b.FA_ERR_ALIGN),
    (dict(lse=P + 2), b.FA_ERR_ALIGN),
    (dict(scale=float("nan")), b.FA_ERR_SCALE),
    (dict(scale=float("inf")), b.FA_ERR_SCALE),
    (dict(scale=0.0), b.FA_ERR_SCALE), (dict(scale=-0.125), b.FA_ERR_SCALE),
])
def test_host_side_argument_checks(kw, code):
    assert call(**kw) == code


def call_qk(q=P, k=P, v=P, o=P, lse=P, B=1, H=1, Nq=128, Nk=64, d=64, causal=1,
            scale=0.125, dtype=b.FA_BF16):
    return b.fa_fwd_qk_raw(q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale,
                           dtype, ctypes.c_void_p(0))


@pytest.mark.parametrize("kw,code", [
    (dict(Nq=-1), b.FA_ERR_SHAPE), (dict(Nk=-1), b.FA_ERR_SHAPE),
    (dict(k=NULL), b.FA_ERR_NULL), (dict(v=NULL), b.FA_ERR_NULL),
    (dict(q=NULL), b.FA_ERR_NULL), (dict(k=P + 4), b.FA_ERR_ALIGN),
    (dict(d=80), b.FA_ERR_HEADDIM), (dict(dtype=5), b.FA_ERR_DTYPE),
    (dict(scale=-1.0), b.FA_ERR_SCALE),
])
def test_host_side_checks_qk(kw, code):
    assert call_qk(**kw) == code


def call_host(q=P, k=P, v=P, o=P, lse=P, qd=P, kd=P, vd=P, od=P, ld=P, B=1, H=1,
              N=128, d=64, causal=0, scale=0.125, dtype=b.FA_BF16):
    return b.fa_fwd_host_raw(q, k, v, o, lse, qd, kd, vd, od, ld, B, H, N, d,
                             causal, scale, dtype, ctypes.c_void_p(0))


@pytest.mark.parametrize("kw,code", [
    (dict(q=NULL), b.FA_ERR_NULL), (dict(o=NULL), b.FA_ERR_NULL),
    (dict(lse=NULL), b.FA_ERR_NULL), (dict(vd=NULL), b.FA_ERR_NULL),
    (dict(ld=NULL), b.FA_ERR_NULL), (dict(B=-1), b.FA_ERR_SHAPE),
    (dict(d=96), b.FA_ERR_HEADDIM), (dict(dtype=2), b.FA_ERR_DTYPE),
    (dict(scale=0.0), b.FA_ERR_SCALE), (dict(kd=P + 8), b.FA_ERR_ALIGN),
    (dict(ld=P + 2), b.FA_ERR_ALIGN),
])
def test_host_side_checks_host_buffers(kw, code):
    assert call_host(**kw) == code


def test_empty_problems_launch_nothing():
    # B, H or N equal to zero is an empty problem: FA_OK, nothing enqueued,
    # pointers never looked at.
    for kw in (dict(B=0), dict(H=0), dict(N=0)):
        assert call(q=NULL, k=NULL, v=NULL, o=NULL, lse=NULL, **kw) == b.FA_OK
    for kw in (dict(B=0), dict(H=0), dict(Nq=0)):
        assert call_qk(q=NULL, k=NULL, v=NULL, o=NULL, lse=NULL, **kw) == b.FA_OK
    for kw in (dict(B=0), dict(H=0), dict(N=0)):
        assert call_host(q=NULL, qd=NULL, o=NULL, ld=NULL, **kw) == b.FA_OK


@pytest.mark.skipif(torch.cuda.is_available(), reason="needs a machine without a GPU")
def test_no_cpu_fallback_without_gpu():
    # Valid arguments but no CUDA device: the call must fail, not compute.
    assert call() == b.FA_ERR_CUDA
    assert call_host() == b.FA_ERR_CUDA
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fwd(q, q, q)


def test_python_wrapper_validation():
    q = torch.zeros(1, 1, 128, 64, dtype=torch.float32)
    with pytest.raises(ValueError):
        fa.fwd(q, q, q[:, :, :64])
    with pytest.raises(TypeError):
        fa.fwd(q, q, q.half())
    with pytest.raises(ValueError):
        fa.fwd(q, q[:, :, :, :32], q[:, :, :, :32])


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        b.load_library(str(tmp_path / "libfa_missing.so"))


def _declared_arities():
    """Parameter count of every function include/*.h declares."""
    out = {}
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", fn)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"FA_API\s+[\w\s\*]+?\b(fa_\w+)\s*\(([^)]*)\)\s*;", src):
            params = m.group(2).strip()
            out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_argument_lists_match_the_header():
    # every ctypes prototype the binding sets up has the header's arity
    lib = fa.load_library()
    arities = _declared_arities()
    assert arities, "no declarations found"
    for name, n in arities.items():
        fn = getattr(lib, name)
        if fn.argtypes is not None:
            assert len(fn.argtypes) == n, (name, len(fn.argtypes), n)
    assert arities["fa_fwd"] == 13 and arities["fa_fwd_host"] == 18
