"""Backward parity: fa_bwd against the fp64 backward oracle.

The backward is checked in isolation on exact forward results: o is the
oracle's O rounded to the dtype and lse the oracle's LSE in fp32, so the only
differences come from the kernel's own arithmetic.  Tolerance, derived from
it (u: unit roundoff of the dtype, 2^-8 for bf16 and 2^-11 for fp16):
  P is recomputed in fp32 (exact products, fp32 LSE) and rounded to the
  dtype for dV = P^T dO:            |d dV| <= u P^T |dO|
  D = rowsum(dO .* o) uses the rounded o:   |dD_i| <= u sum_t |dO_it o_it|
  dS = P (dP - D) is rounded to the dtype:
        |d dS_ij| <= u |dS_ij| + P_ij |dD_i|
  dK = scale dS^T Q, dQ = scale dS K:  |d dK| <= scale |d dS|^T |Q| etc.
  and every output is rounded once more (u |ref|).
The test allows twice those bounds plus 1e-5 * max |ref| for fp32
accumulation.  The bound's terms are evaluated with numpy from the oracle's
probabilities; the reference values themselves come from the C oracle.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_39_gb300 as fa
from exact_attention_39_gb300 import binding as b
from exact_attention_39_gb300 import workloads as W
import oracle

U = {"bf16": 2.0 ** -8, "fp16": 2.0 ** -11}


def softmax_probs(q, k, scale, causal):
    s = scale * np.einsum("...id,...jd->...ij", q, k)
    nq, nk = q.shape[-2], k.shape[-2]
    if causal:
        vis = np.arange(nk)[None, :] <= (np.arange(nq)[:, None] + nk - nq)
        s = np.where(vis, s, -np.inf)
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=-1, keepdims=True)


def run_and_check(w, o_from="oracle"):
    q, k, v = W.make_inputs(w)
    g = W.make_upstream_grad(w)
    dt = W.DTYPES[w.dtype]
    q64, k64, v64, g64 = (t.double().numpy() for t in (q, k, v, g))
    o_ref, lse_ref = oracle.attention_fwd(q64, k64, v64, w.scale, w.causal)
    dev = torch.device("cuda")
    if o_from == "oracle":
        o = torch.from_numpy(o_ref).to(dt)
        lse = torch.from_numpy(lse_ref).float()
    else:   # the GPU forward's own outputs
        o, lse = fa.fwd(q.to(dev), k.to(dev), v.to(dev), causal=w.causal, scale=w.scale)
        o, lse = o.cpu(), lse.cpu()
    dq, dk, dv = fa.bwd(*(t.to(dev) for t in (q, k, v, o, lse, g)),
                        causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    o64 = o.double().numpy()
    rq, rk, rv = oracle.attention_bwd(q64, k64, v64, g64, w.scale, w.causal)
    # tolerance terms
    u = U[w.dtype]
    P = softmax_probs(q64, k64, w.scale, w.causal)
    dP = np.einsum("...id,...jd->...ij", g64, v64)
    D = (g64 * o_ref).sum(-1)
    dS = P * (dP - D[..., None])
    dD = u * np.abs(g64 * o64).sum(-1) + np.abs((g64 * (o64 - o_ref)).sum(-1))
    eS = u * np.abs(dS) + P * dD[..., None]
    bound = {
        "dv": u * np.einsum("...ij,...id->...jd", P, np.abs(g64)) + u * np.abs(rv),
        "dk": w.scale * np.einsum("...ij,...id->...jd", eS, np.abs(q64)) + u * np.abs(rk),
        "dq": w.scale * np.einsum("...ij,...jd->...id", eS, np.abs(k64)) + u * np.abs(rq),
    }
    got = {"dq": dq.cpu().double().numpy(), "dk": dk.cpu().double().numpy(),
           "dv": dv.cpu().double().numpy()}
    ref = {"dq": rq, "dk": rk, "dv": rv}
    for name in ("dq", "dk", "dv"):
        err = np.abs(got[name] - ref[name])
        tol = 2 * bound[name] + 1e-5 * np.abs(ref[name]).max()
        worst = (err - tol).max()
        assert np.isfinite(got[name]).all(), name
        assert worst <= 0, "%s %s: max err %.3g, worst excess %.3g, max |ref| %.3g" % (
            w.name, name, err.max(), worst, np.abs(ref[name]).max())


@pytest.mark.gpu
@pytest.mark.parametrize("n", [128, 256, 300, 1000])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d,dtype", [(64, "bf16"), (64, "fp16"), (128, "bf16"), (128, "fp16")])
def test_bwd_parity(n, causal, d, dtype):
    w = W.Workload("bwd", 1, 2, n, d, dtype, causal, seed=n + d)
    run_and_check(w)


@pytest.mark.gpu
@pytest.mark.parametrize("n", [1, 5, 127, 129])
def test_bwd_small_and_ragged(n):
    run_and_check(W.Workload("bwd_small", 2, 2, n, 64, "bf16", True, seed=n))


@pytest.mark.gpu
def test_bwd_after_gpu_forward():
    # the gradients from the GPU forward's own O and LSE (the usual use)
    run_and_check(W.Workload("bwd_e2e", 1, 4, 640, 64, "bf16", True, seed=3),
                  o_from="gpu")


@pytest.mark.gpu
def test_bwd_matches_torch_autograd_direction():
    # d/deps L(q + eps u) at eps = 0 equals <dQ, u> (directional derivative,
    # evaluated with the oracle forward in fp64)
    w = W.Workload("bwd_dir", 1, 1, 200, 64, "bf16", True, seed=11)
    q, k, v = W.make_inputs(w)
    g = W.make_upstream_grad(w)
    dev = torch.device("cuda")
    o, lse = fa.fwd(q.to(dev), k.to(dev), v.to(dev), causal=True)
    dq, _, _ = fa.bwd(q.to(dev), k.to(dev), v.to(dev), o, lse, g.to(dev), causal=True)
    q64, k64, v64, g64 = (t.double().numpy() for t in (q, k, v, g))
    u = np.random.default_rng(0).standard_normal(q64.shape)
    eps = 1e-4
    lp = (oracle.attention_fwd(q64 + eps * u, k64, v64, w.scale, True)[0] * g64).sum()
    lm = (oracle.attention_fwd(q64 - eps * u, k64, v64, w.scale, True)[0] * g64).sum()
    num = (lp - lm) / (2 * eps)
    ana = float((dq.cpu().double().numpy() * u).sum())
    assert abs(num - ana) <= 2e-2 * abs(num) + 1e-3


# ---------------------------------------------------------------- host side
def test_bwd_workspace_size_and_checks():
    # two fp32 per query row, each head padded to whole 128-row blocks
    assert fa.bwd_workspace_bytes(1, 1, 1) == 2 * 128 * 4
    assert fa.bwd_workspace_bytes(1, 1, 129) == 2 * 256 * 4
    assert fa.bwd_workspace_bytes(8, 32, 8192) == 2 * 8 * 32 * 8192 * 4
    assert fa.bwd_workspace_bytes(0, 1, 1) == 0
    P = 0x10000
    import ctypes
    args = lambda **kw: dict(dict(ws=P, wsb=1 << 20, N=128, d=64, dtype=b.FA_BF16,
                                  scale=0.125), **kw)

    def call(**kw):
        a = args(**kw)
        return b.fa_bwd_raw(P, P, P, P, P, P, P, P, P, a["ws"], a["wsb"], 1, 1, a["N"],
                            a["d"], 1, a["scale"], a["dtype"], ctypes.c_void_p(0))
    assert call(ws=0) == b.FA_ERR_WORKSPACE
    assert call(wsb=16) == b.FA_ERR_WORKSPACE
    assert call(wsb=2 * 128 * 4 - 4) == b.FA_ERR_WORKSPACE
    assert call(ws=P + 4) == b.FA_ERR_WORKSPACE
    assert call(d=96) == b.FA_ERR_HEADDIM
    assert call(dtype=7) == b.FA_ERR_DTYPE
    assert call(scale=-1.0) == b.FA_ERR_SCALE
    assert call(N=-1) == b.FA_ERR_SHAPE
    assert call(N=0, ws=0) == b.FA_OK
