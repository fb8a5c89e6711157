"""ctypes binding of the C ABI in include/fa.h.

Argument marshalling only: every step of the attention forward runs in the
CUDA kernel behind ``fa_fwd``.  PyTorch supplies device memory and streams.
There is no fallback: if the shared library is missing or the call fails,
these functions raise.
"""
import ctypes
import math
import os

import torch

from . import _build

FA_OK = 0
FA_ERR_NULL = 1
FA_ERR_SHAPE = 2
FA_ERR_HEADDIM = 3
FA_ERR_DTYPE = 4
FA_ERR_ALIGN = 5
FA_ERR_SCALE = 6
FA_ERR_CUDA = 7
FA_ERR_DEVICE_TIMEOUT = 8
FA_ERR_WORKSPACE = 9
FA_FP16 = 0
FA_BF16 = 1

EXPORTED = ("fa_fwd", "fa_fwd_qk", "fa_fwd_fp8", "fa_fwd_host", "fa_bwd", "fa_bwd_workspace_bytes",
            "fa_bwd_noalloc", "fa_status_string", "fa_last_device_error",
            "fa_version", "fa_selftest_wait_timeout")
FA_BWD_NOALLOC_MAX_ROWS = 1 << 21

_lib = None


class FaError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__("%s (status %d)" % (msg, status))
        self.status = status


def load_library(path=None):
    """Load libfa_sm103.so (built in-tree by ``_build.build``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or _build.LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(
            "%s is not built; run `python -c \"import __graft_entry__ as g; "
            "g.build()\"` first (there is no CPU fallback)" % path)
    lib = ctypes.CDLL(path)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    lib.fa_fwd.restype = i
    lib.fa_fwd_qk.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
    lib.fa_fwd_qk.restype = i
    lib.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, f, f, f, vp]
    lib.fa_fwd_fp8.restype = i
    lib.fa_fwd_host.argtypes = [vp] * 10 + [i, i, i, i, i, f, i, vp]
    lib.fa_fwd_host.restype = i
    sz = ctypes.c_size_t
    lib.fa_bwd_workspace_bytes.argtypes = [i, i, i]
    lib.fa_bwd_workspace_bytes.restype = sz
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i,
                           i, f, i, vp]
    lib.fa_bwd.restype = i
    lib.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i,
                                   i, f, i, vp]
    lib.fa_bwd_noalloc.restype = i
    lib.fa_selftest_wait_timeout.argtypes = [ctypes.c_ulonglong, vp]
    lib.fa_selftest_wait_timeout.restype = i
    lib.fa_status_string.argtypes = [i]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_last_device_error.argtypes = [vp]
    lib.fa_last_device_error.restype = i
    lib.fa_version.argtypes = []
    lib.fa_version.restype = i
    if path == _build.LIB_PATH:
        _lib = lib
    return lib


def status_string(status):
    return load_library().fa_status_string(int(status)).decode()


def _check(status):
    if status != FA_OK:
        raise FaError(status, status_string(status))


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _require_on(device, what, *tensors):
    """Every tensor a contiguous CUDA tensor on ``device``: the library runs on
    the current device and dereferences every pointer there."""
    for t in tensors:
        if not t.is_cuda or t.device != device or not t.is_contiguous():
            raise ValueError("%s must be contiguous CUDA tensors on %s" % (what, device))


def _require_stream_on(device, stream):
    if stream is not None and stream.device != device:
        raise ValueError("stream is on %s, the tensors on %s" % (stream.device, device))


def fa_fwd_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, N, d, causal,
               scale, dtype_code, stream_handle):
    """The C call with plain integers; returns the status code."""
    return load_library().fa_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, int(B),
                                 int(H), int(N), int(d), int(bool(causal)),
                                 float(scale), int(dtype_code), stream_handle)


def fa_fwd_qk_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, Nq, Nk, d,
                  causal, scale, dtype_code, stream_handle):
    """The C call for different query and key lengths; returns the status."""
    return load_library().fa_fwd_qk(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr,
                                    int(B), int(H), int(Nq), int(Nk), int(d),
                                    int(bool(causal)), float(scale),
                                    int(dtype_code), stream_handle)


def fa_fwd_fp8_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, Nq, Nk, d,
                   causal, scale, q_descale, k_descale, v_descale,
                   stream_handle):
    """The C call of the e4m3 forward; returns the status."""
    return load_library().fa_fwd_fp8(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr,
                                     int(B), int(H), int(Nq), int(Nk), int(d),
                                     int(bool(causal)), float(scale),
                                     float(q_descale), float(k_descale),
                                     float(v_descale), stream_handle)


def _dtype_code(t):
    if t.dtype == torch.float16:
        return FA_FP16
    if t.dtype == torch.bfloat16:
        return FA_BF16
    raise TypeError("q, k, v must be float16 or bfloat16, got %s" % t.dtype)


def fwd(q, k, v, causal=False, scale=None, out=None, lse=None, stream=None):
    """Attention forward on CUDA tensors q [B, H, Nq, d], k and v [B, H, Nk, d].

    Returns ``(o, lse)``: ``o`` like ``q``; ``lse`` [B, H, Nq] float32.
    With Nq != Nk the causal mask is aligned to the bottom-right corner
    (key j visible to query i iff j <= i + Nk - Nq).  ``scale`` defaults to
    1/sqrt(d).  The kernel is enqueued on ``stream`` (default: the current
    torch stream); nothing is synchronised.
    """
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("q must be [B, H, Nq, d] and k, v [B, H, Nk, d]")
    if k.shape[:2] != q.shape[:2] or k.shape[3] != q.shape[3]:
        raise ValueError("q, k, v must agree in B, H and d")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    code = _dtype_code(q)
    if not q.is_cuda:
        raise ValueError("q, k, v must be contiguous CUDA tensors")
    _require_on(q.device, "q, k, v", q, k, v)
    _require_stream_on(q.device, stream)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("out must be a contiguous tensor like q")
    if lse.shape != (B, H, Nq) or lse.dtype != torch.float32:
        raise ValueError("lse must be a contiguous float32 [B, H, Nq] tensor")
    _require_on(q.device, "out and lse", out, lse)
    with torch.cuda.device(q.device):
        if Nq == Nk:
            st = fa_fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                            out.data_ptr(), lse.data_ptr(), B, H, Nq, d,
                            causal, scale, code, _stream_handle(stream))
        else:
            st = fa_fwd_qk_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                               out.data_ptr(), lse.data_ptr(), B, H, Nq, Nk, d,
                               causal, scale, code, _stream_handle(stream))
        _check(st)
    return out, lse


def fwd_fp8(q, k, v, q_descale, k_descale, v_descale, causal=False,
            scale=None, out=None, lse=None, stream=None):
    """Attention forward on float8_e4m3fn CUDA tensors (real values are
    q * q_descale etc.); returns ``(o, lse)`` with ``o`` bf16 [B, H, Nq, d]."""
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("q must be [B, H, Nq, d] and k, v [B, H, Nk, d]")
    if k.shape[:2] != q.shape[:2] or k.shape[3] != q.shape[3]:
        raise ValueError("q, k, v must agree in B, H and d")
    for t in (q, k, v):
        if t.dtype != torch.float8_e4m3fn:
            raise TypeError("q, k, v must be torch.float8_e4m3fn")
    if not q.is_cuda:
        raise ValueError("q, k, v must be contiguous CUDA tensors")
    _require_on(q.device, "q, k, v", q, k, v)
    _require_stream_on(q.device, stream)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if out.shape != (B, H, Nq, d) or out.dtype != torch.bfloat16:
        raise ValueError("out must be a contiguous bf16 [B, H, Nq, d] tensor")
    if lse.shape != (B, H, Nq) or lse.dtype != torch.float32:
        raise ValueError("lse must be a contiguous float32 [B, H, Nq] tensor")
    _require_on(q.device, "out and lse", out, lse)
    with torch.cuda.device(q.device):
        _check(fa_fwd_fp8_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                              out.data_ptr(), lse.data_ptr(), B, H, Nq, Nk, d,
                              causal, scale, q_descale, k_descale, v_descale,
                              _stream_handle(stream)))
    return out, lse


def bwd_workspace_bytes(B, H, N):
    return int(load_library().fa_bwd_workspace_bytes(int(B), int(H), int(N)))


def fa_bwd_raw(q_ptr, k_ptr, v_ptr, o_ptr, do_ptr, lse_ptr, dq_ptr, dk_ptr,
               dv_ptr, ws_ptr, ws_bytes, B, H, N, d, causal, scale, dtype_code,
               stream_handle):
    """The C call of the backward; returns the status."""
    return load_library().fa_bwd(q_ptr, k_ptr, v_ptr, o_ptr, do_ptr, lse_ptr,
                                 dq_ptr, dk_ptr, dv_ptr, ws_ptr, int(ws_bytes),
                                 int(B), int(H), int(N), int(d),
                                 int(bool(causal)), float(scale),
                                 int(dtype_code), stream_handle)


def fa_bwd_noalloc_raw(q_ptr, k_ptr, v_ptr, o_ptr, do_ptr, lse_ptr, dq_ptr,
                       dk_ptr, dv_ptr, B, H, N, d, causal, scale, dtype_code,
                       stream_handle):
    """The C call of the backward that uses the library's static scratch
    instead of a workspace (for callers that cannot allocate); returns the
    status."""
    return load_library().fa_bwd_noalloc(q_ptr, k_ptr, v_ptr, o_ptr, do_ptr,
                                         lse_ptr, dq_ptr, dk_ptr, dv_ptr,
                                         int(B), int(H), int(N), int(d),
                                         int(bool(causal)), float(scale),
                                         int(dtype_code), stream_handle)


def bwd(q, k, v, o, lse, dout, causal=False, scale=None, dq=None, dk=None,
        dv=None, workspace=None, stream=None):
    """Gradients (dq, dk, dv) of the attention forward for the upstream
    gradient ``dout`` of ``o``.  All [B, H, N, d] CUDA tensors of one dtype
    (``lse`` [B, H, N] float32, as ``fwd`` returned them).  ``workspace``
    (a CUDA uint8 tensor of at least ``bwd_workspace_bytes`` bytes) is
    allocated when not given."""
    if q.dim() != 4 or any(t.shape != q.shape for t in (k, v, o, dout)):
        raise ValueError("q, k, v, o, dout must all be [B, H, N, d]")
    if not (q.dtype == k.dtype == v.dtype == o.dtype == dout.dtype):
        raise TypeError("q, k, v, o, dout must share one dtype")
    code = _dtype_code(q)
    if not q.is_cuda:
        raise ValueError("inputs must be contiguous CUDA tensors")
    _require_on(q.device, "inputs", q, k, v, o, dout, lse)
    _require_stream_on(q.device, stream)
    B, H, N, d = q.shape
    if lse.shape != (B, H, N) or lse.dtype != torch.float32:
        raise ValueError("lse must be a float32 [B, H, N] tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t in (dq, dk, dv):
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError("dq, dk, dv must be contiguous tensors like q")
    _require_on(q.device, "dq, dk, dv", dq, dk, dv)
    need = bwd_workspace_bytes(B, H, N)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _require_on(q.device, "workspace", workspace)
    with torch.cuda.device(q.device):
        _check(fa_bwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                          dout.data_ptr(), lse.data_ptr(), dq.data_ptr(),
                          dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(),
                          workspace.numel() * workspace.element_size(), B, H, N,
                          d, causal, scale, code, _stream_handle(stream)))
    return dq, dk, dv


def fa_fwd_host_raw(q_h, k_h, v_h, o_h, lse_h, q_d, k_d, v_d, o_d, lse_d,
                    B, H, N, d, causal, scale, dtype_code, stream_handle):
    """The C call with plain integers; returns the status code."""
    return load_library().fa_fwd_host(q_h, k_h, v_h, o_h, lse_h, q_d, k_d, v_d,
                                      o_d, lse_d, int(B), int(H), int(N), int(d),
                                      int(bool(causal)), float(scale),
                                      int(dtype_code), stream_handle)


def fwd_host(q_h, k_h, v_h, q_d, k_d, v_d, o_d, lse_d, o_h, lse_h,
             causal=False, scale=None, stream=None):
    """End-to-end call from host memory through ``fa_fwd_host``: q, k, v
    (pinned host tensors) go up through the device staging buffers, O and LSE
    come back into the pinned host tensors ``o_h``/``lse_h``; the library
    overlaps the copies with the kernel chunk by chunk.  Returns after
    synchronising ``stream``."""
    for t in (q_h, k_h, v_h, o_h, lse_h):
        if t.device.type != "cpu" or not t.is_contiguous():
            raise ValueError("host tensors must be contiguous CPU tensors")
    if not q_d.is_cuda:
        raise ValueError("staging tensors must be contiguous CUDA tensors")
    _require_on(q_d.device, "staging tensors", q_d, k_d, v_d, o_d, lse_d)
    _require_stream_on(q_d.device, stream)
    if q_h.dim() != 4 or k_h.shape != q_h.shape or v_h.shape != q_h.shape:
        raise ValueError("q, k, v must share one [B, H, N, d] shape")
    for a, b in ((q_h, q_d), (k_h, k_d), (v_h, v_d), (o_h, o_d), (lse_h, lse_d)):
        if a.shape != b.shape or a.dtype != b.dtype:
            raise ValueError("host and staging tensors disagree in shape or dtype")
    if o_h.shape != q_h.shape or o_h.dtype != q_h.dtype:
        raise ValueError("o must match q")
    B, H, N, d = q_h.shape
    if lse_h.shape != (B, H, N) or lse_h.dtype != torch.float32:
        raise ValueError("lse must be float32 [B, H, N]")
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    with torch.cuda.device(q_d.device):
        stream = stream or torch.cuda.current_stream()
        _check(fa_fwd_host_raw(q_h.data_ptr(), k_h.data_ptr(), v_h.data_ptr(),
                               o_h.data_ptr(), lse_h.data_ptr(), q_d.data_ptr(),
                               k_d.data_ptr(), v_d.data_ptr(), o_d.data_ptr(),
                               lse_d.data_ptr(), B, H, N, d, causal, scale,
                               _dtype_code(q_h), _stream_handle(stream)))
    stream.synchronize()
    return o_h, lse_h


def last_device_error(stream=None):
    """Synchronise and return the device status (FA_OK or an error code)."""
    return load_library().fa_last_device_error(_stream_handle(stream))


def version():
    return load_library().fa_version()


def selftest_wait_timeout(timeout_ns, stream=None):
    """Enqueue the bounded-wait self-test kernel; returns the launch status."""
    return load_library().fa_selftest_wait_timeout(int(timeout_ns),
                                                   _stream_handle(stream))
