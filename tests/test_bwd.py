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
When o and lse come from the GPU forward (the benchmarked shapes, and the
usual use), P inherits the error of the given LSE: P_gpu = P exp(lse_ref -
lse_gpu), so |dP| <= P expm1(|d lse|) adds to dV through P^T |dO| and to dS
through |dP - D|.
The test allows twice those bounds plus 1e-5 * max |ref| for fp32
accumulation.  The bound's terms are evaluated with numpy from the oracle's
exact LSE, in row chunks (no N x N matrix is held), on every row and key or on
sampled ones; the reference values themselves come from the C oracle.
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


def _probs_block(q, k, lse_ref, scale, causal, rows, keys, nq, nk):
    """P[rows][:, keys] of one head from the exact LSE (masked entries 0)."""
    s = scale * (q[rows] @ k[keys].T)
    p = np.exp(s - lse_ref[rows][:, None])
    if causal:
        p = np.where(keys[None, :] <= rows[:, None] + nk - nq, p, 0.0)
    return p


def bwd_bounds(q, k, v, g, o_gpu, lse_gpu, o_ref, lse_ref, scale, causal, u,
               rows=None, keys=None, chunk=512):
    """Per-element error bounds (before the output rounding) of dQ on query
    ``rows`` and of dK, dV on ``keys`` (all when None) for one head, from the
    terms in the module docstring plus the error the kernel's P inherits
    from the LSE it is given: P_gpu = P exp(lse_ref - lse_gpu).
    Computed in row chunks so that no N x N matrix is held."""
    nq, nk = q.shape[0], k.shape[0]
    rows = np.arange(nq) if rows is None else np.asarray(rows)
    keys = np.arange(nk) if keys is None else np.asarray(keys)
    D = (g * o_ref).sum(-1)
    dD = u * np.abs(g * o_gpu).sum(-1) + np.abs((g * (o_gpu - o_ref)).sum(-1))
    dl = np.expm1(np.abs(lse_gpu - lse_ref))

    def terms(r, kk):
        p = _probs_block(q, k, lse_ref, scale, causal, r, kk, nq, nk)
        dp = g[r] @ v[kk].T - D[r][:, None]          # dP - D
        ep = p * dl[r][:, None]                       # from the given LSE
        es = u * np.abs(p * dp) + p * dD[r][:, None] + ep * np.abs(dp)
        return p, ep, es

    bq = np.zeros((rows.size, q.shape[1]))
    for c0 in range(0, rows.size, chunk):
        r = rows[c0:c0 + chunk]
        _, _, es = terms(r, np.arange(nk))
        bq[c0:c0 + chunk] = scale * (es @ np.abs(k))
    bk = np.zeros((keys.size, q.shape[1]))
    bv = np.zeros((keys.size, q.shape[1]))
    for c0 in range(0, nq, chunk):
        r = np.arange(c0, min(nq, c0 + chunk))
        p, ep, es = terms(r, keys)
        bv += (u * p + ep).T @ np.abs(g[r])
        bk += scale * (es.T @ np.abs(q[r]))
    return bq, bk, bv


def check_head(name, got, ref, bounds, u):
    """got/ref: dicts of dq, dk, dv (already restricted to the checked rows
    and keys); bounds: (bq, bk, bv) from bwd_bounds."""
    for key, bnd in zip(("dq", "dk", "dv"), bounds):
        r = ref[key]
        err = np.abs(got[key] - r)
        tol = 2 * (bnd + u * np.abs(r)) + 1e-5 * np.abs(r).max()
        worst = (err - tol).max()
        assert np.isfinite(got[key]).all(), (name, key)
        assert worst <= 0, "%s %s: max err %.3g, worst excess %.3g, max |ref| %.3g" % (
            name, key, err.max(), worst, np.abs(r).max())


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
    o64, l64 = o.double().numpy(), lse.double().numpy()
    rq, rk, rv = oracle.attention_bwd(q64, k64, v64, g64, w.scale, w.causal)
    u = U[w.dtype]
    got = [t.cpu().double().numpy() for t in (dq, dk, dv)]
    for b_ in range(w.B):
        for h in range(w.H):
            at = lambda a: a[b_, h]
            bounds = bwd_bounds(at(q64), at(k64), at(v64), at(g64), at(o64), at(l64),
                                at(o_ref), at(lse_ref), w.scale, w.causal, u)
            check_head("%s[%d,%d]" % (w.name, b_, h),
                       {"dq": at(got[0]), "dk": at(got[1]), "dv": at(got[2])},
                       {"dq": at(rq), "dk": at(rk), "dv": at(rv)}, bounds, u)


def run_and_check_sampled(w, n_heads, rows=None, keys=None):
    """The benchmarked shapes: the whole workload through the GPU forward and
    fa_bwd exactly as the benchmark launches them, then ``n_heads`` sampled
    (b, h) slices against the oracle (on sampled query rows and keys when
    given)."""
    dev = torch.device("cuda")
    q, k, v = W.make_inputs(w)
    g = W.make_upstream_grad(w)
    qd, kd, vd, gd = (t.to(dev) for t in (q, k, v, g))
    o, lse = fa.fwd(qd, kd, vd, causal=w.causal, scale=w.scale)
    ws = torch.empty(fa.bwd_workspace_bytes(w.B, w.H, w.N), dtype=torch.uint8, device=dev)
    dq, dk, dv = fa.bwd(qd, kd, vd, o, lse, gd, causal=w.causal, scale=w.scale, workspace=ws)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    u = U[w.dtype]
    for b_, h in W.sample_heads(w, n_heads):
        at = lambda t: t[b_, h].double().cpu().numpy()
        q64, k64, v64, g64 = at(q), at(k), at(v), at(g)
        o_ref, lse_ref = oracle.attention_fwd(q64, k64, v64, w.scale, w.causal)
        rq, rk, rv = oracle.attention_bwd(q64, k64, v64, g64, w.scale, w.causal)
        bounds = bwd_bounds(q64, k64, v64, g64, at(o), at(lse), o_ref, lse_ref, w.scale,
                            w.causal, u, rows=rows, keys=keys)
        sel_r = slice(None) if rows is None else np.asarray(rows)
        sel_k = slice(None) if keys is None else np.asarray(keys)
        check_head("%s[%d,%d]" % (w.name, b_, h),
                   {"dq": at(dq)[sel_r], "dk": at(dk)[sel_k], "dv": at(dv)[sel_k]},
                   {"dq": rq[sel_r], "dk": rk[sel_k], "dv": rv[sel_k]}, bounds, u)


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
@pytest.mark.parametrize("n", [63, 64, 65, 191, 193])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_bwd_inner_block_boundaries(n, causal, d):
    # both kernels loop over 64-row inner blocks (query blocks in the dK/dV
    # kernel, key blocks in the dQ kernel): lengths just below, at and above
    # a multiple of 64, so that the last block is partial, full, or one row
    run_and_check(W.Workload("bwd_blk", 1, 2, n, d, "bf16", causal, seed=3 * n + d))


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_d128_many_blocks(causal):
    # d = 128 (predicated MMA issue, two S/dP buffers, four-stage rings):
    # 32 inner blocks per CTA, every row and key of two heads checked
    run_and_check(W.Workload("bwd_d128", 1, 2, 2048, 128, "bf16", causal, seed=21,
                             in_mult=0.5))


@pytest.mark.gpu
@pytest.mark.parametrize("d", [64, 128])
def test_bwd_deterministic(d):
    # no atomics and a fixed order of every sum: a second call on the same
    # inputs gives the same bits (d = 64 and d = 128 issue their MMAs in the
    # two different forms)
    w = W.Workload("bwd_det", 2, 3, 777, d, "bf16", True, seed=11 + d)
    dev = torch.device("cuda")
    q, k, v = (t.to(dev) for t in W.make_inputs(w))
    g = W.make_upstream_grad(w).to(dev)
    o, lse = fa.fwd(q, k, v, causal=w.causal, scale=w.scale)
    first = fa.bwd(q, k, v, o, lse, g, causal=w.causal, scale=w.scale)
    second = fa.bwd(q, k, v, o, lse, g, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    for a, b_ in zip(first, second):
        assert torch.equal(a, b_)
        assert torch.isfinite(a.float()).all()


@pytest.mark.gpu
@pytest.mark.parametrize("w", [W.N2048, W.N2048_CAUSAL, W.N8192, W.N8192_CAUSAL],
                         ids=lambda w: w.name)
def test_bwd_benchmark_shapes_d64(w):
    # B8 H32 d64 bf16 at N = 2048 and 8192: 16 and 64 key blocks per CTA,
    # 4096 and 16384 CTAs per kernel; 2 sampled heads, every row and key
    run_and_check_sampled(w, n_heads=2)


@pytest.mark.gpu
def test_bwd_long_context_d128_causal():
    # B1 H32 N32768 d128 bf16 causal (inputs N(0,1)/2): 256 query blocks;
    # one sampled head, 256 sampled query rows and 256 sampled keys
    w = W.LONG
    sel = W.sample_rows(w.N, 256)
    run_and_check_sampled(w, n_heads=1, rows=sel, keys=sel)


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


def test_chunked_bounds_equal_the_dense_formulas():
    # bwd_bounds (row chunks, sampled rows/keys) against the same terms
    # written densely with full N x N matrices, on a small head
    rng = np.random.default_rng(5)
    nq = nk = 70
    d, scale, u = 8, 0.3, 2.0 ** -8
    q, k, v, g = (rng.standard_normal((n, d)) for n in (nq, nk, nk, nq))
    for causal in (False, True):
        o_ref, lse_ref = oracle.attention_fwd(q, k, v, scale, causal)
        o_gpu = o_ref + 1e-3 * rng.standard_normal(o_ref.shape)
        lse_gpu = lse_ref + 1e-4 * rng.standard_normal(lse_ref.shape)
        P = softmax_probs(q, k, scale, causal)
        dp = g @ v.T - (g * o_ref).sum(-1)[:, None]
        dD = u * np.abs(g * o_gpu).sum(-1) + np.abs((g * (o_gpu - o_ref)).sum(-1))
        ep = P * np.expm1(np.abs(lse_gpu - lse_ref))[:, None]
        es = u * np.abs(P * dp) + P * dD[:, None] + ep * np.abs(dp)
        dense = (scale * es @ np.abs(k), scale * es.T @ np.abs(q),
                 (u * P + ep).T @ np.abs(g))
        rows, keys = np.array([0, 3, 69]), np.array([1, 2, 40, 69])
        for r, kk, ch in ((None, None, 16), (rows, keys, 7)):
            got = bwd_bounds(q, k, v, g, o_gpu, lse_gpu, o_ref, lse_ref, scale, causal,
                             u, rows=r, keys=kk, chunk=ch)
            sr = slice(None) if r is None else r
            sk = slice(None) if kk is None else kk
            np.testing.assert_allclose(got[0], dense[0][sr], rtol=1e-12, atol=1e-300)
            np.testing.assert_allclose(got[1], dense[1][sk], rtol=1e-12, atol=1e-300)
            np.testing.assert_allclose(got[2], dense[2][sk], rtol=1e-12, atol=1e-300)
