"""FP8 (e4m3) forward against the fp64 oracle on the dequantized inputs.

Tolerance, derived from the arithmetic: the two products are exact in
fp32 up to accumulation rounding; the one coarse step is P rounded to e4m3
before P V, while the row sum l uses the fp32 probabilities.  e4m3 rounding
to nearest errs by at most 2^-4 p for normal values and 2^-10 in the
subnormal range, so |Q(p) - p| <= 2^-4 p + 2^-10 and
    |dO_i| <= 2^-4 attn(Q, K, |V|)_i + 2^-10 sum_j |v_j| / l_i .
The kernel's offset never exceeds the true row maximum, so its largest
probability is >= 1 and l_i >= exp(LSE_i - s_max,i) (s the scaled logits);
the test uses that lower bound.  Added: the bf16 rounding of O (2^-8 |O|,
twice the half-ulp) and 1e-4 for fp32 accumulation and ex2.approx.  The
mean error must stay below 2^-5 * mean attn(|V|) (the roundings are
unbiased); LSE within 1e-3 as for the 16-bit path.
"""
import ctypes

import numpy as np
import pytest
import torch

import exact_attention_39_gb300 as fa
from exact_attention_39_gb300 import binding as b
from exact_attention_39_gb300 import workloads as W
import oracle

D = W.E4M3_DESCALE


def run_fp8(w, q, k, v, scale=None):
    dev = torch.device("cuda")
    o, lse = fa.fwd_fp8(q.to(dev), k.to(dev), v.to(dev), D, D, D,
                        causal=w.causal, scale=scale or w.scale)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    return o.cpu(), lse.cpu()


def check_fp8(w, o, lse, q, k, v, heads=None, rows=None, scale=None):
    scale = scale or w.scale
    # dequantise first (fp8 tensors cannot be indexed on the CPU)
    q, k, v = (W.dequantized(t, "e4m3") for t in (q, k, v))
    if heads is not None:
        idx = torch.tensor([bb * w.H + h for bb, h in heads])
        flat = lambda t: t.reshape(w.B * w.H, *t.shape[2:])[idx]
        q, k, v, o, lse = (flat(t) for t in (q, k, v, o, lse))
    qs, ks, vs = q.numpy(), k.numpy(), v.numpy()
    og, lg = o.double().numpy(), lse.double().numpy()
    if rows is not None:
        og, lg = og[..., rows, :], lg[..., rows]
    o_ref, l_ref = oracle.attention_fwd(qs, ks, vs, scale, w.causal, rows=rows)
    a_abs, _ = oracle.attention_fwd(qs, ks, np.abs(vs), scale, w.causal, rows=rows)
    # per row: largest visible scaled logit and the sum of visible |v|
    nq, nk = qs.shape[-2], ks.shape[-2]
    r_idx = np.arange(nq) if rows is None else np.asarray(rows)
    s_all = scale * np.einsum("...id,...jd->...ij", qs[..., r_idx, :], ks)
    vis = np.ones((len(r_idx), nk), dtype=bool)
    if w.causal:
        vis = np.arange(nk)[None, :] <= (r_idx[:, None] + nk - nq)
    s_max = np.where(vis, s_all, -np.inf).max(axis=-1)
    v_sum = np.einsum("ij,...jd->...id", vis.astype(np.float64), np.abs(vs))
    inv_l = np.exp(np.minimum(s_max - l_ref, 0.0))          # 1 / l lower bound
    err = np.abs(og - o_ref)
    tol = (2.0 ** -4 * a_abs + 2.0 ** -10 * v_sum * inv_l[..., None]
           + 2.0 ** -8 * np.abs(o_ref) + 1e-4)
    worst = (err - tol).max()
    msg = "%s: max|dO|=%.3g mean|dO|=%.3g worst excess=%.3g max|dLSE|=%.3g" % (
        w.name, err.max(), err.mean(), worst, np.abs(lg - l_ref).max())
    assert np.isfinite(og).all(), msg
    assert worst <= 0, msg
    assert err.mean() <= 2.0 ** -5 * a_abs.mean(), msg
    assert np.abs(lg - l_ref).max() <= 1e-3, msg


@pytest.mark.gpu
@pytest.mark.parametrize("n,causal,d", [(128, False, 64), (300, True, 64), (1000, False, 64),
                                        (129, True, 128), (500, False, 128), (777, True, 128)])
def test_fp8_small(n, causal, d):
    w = W.Workload("fp8", 2, 3, n, d, "e4m3", causal, seed=n + d)
    q, k, v = W.make_inputs(w)
    o, lse = run_fp8(w, q, k, v)
    check_fp8(w, o, lse, q, k, v)


@pytest.mark.gpu
@pytest.mark.parametrize("nq,nk", [(100, 700), (700, 100), (1, 300)])
def test_fp8_query_key_lengths(nq, nk):
    w = W.Workload("fp8qk", 1, 2, nq, 64, "e4m3", True, seed=nq, Nk=nk)
    q, k, v = W.make_inputs(w)
    o, lse = run_fp8(w, q, k, v)
    dead = max(0, nq - nk)
    assert (o[:, :, :dead] == 0).all()
    check_fp8(w, o, lse, q, k, v, rows=list(range(dead, nq)))


# e4m3 at d = 64 runs one query tile per CTA at every length: ragged query and
# key tails above 4096 keys, where 16-bit inputs switch to two tiles per CTA
@pytest.mark.gpu
@pytest.mark.parametrize("nq,nk,causal", [(300, 5000, False), (300, 5000, True),
                                          (4353, 4353, True), (1, 4200, False)])
def test_fp8_one_tile_long_keys(nq, nk, causal):
    w = W.Workload("fp8long", 1, 2, nq, 64, "e4m3", causal, seed=nq + nk, Nk=nk)
    q, k, v = W.make_inputs(w)
    o, lse = run_fp8(w, q, k, v)
    dead = max(0, nq - nk) if causal else 0
    check_fp8(w, o, lse, q, k, v, rows=list(range(dead, nq)))


@pytest.mark.gpu
def test_fp8_large_logits():
    # logits eight times larger, through the softmax scale (multiplying Q by
    # 8 would leave e4m3's range at this descale)
    w = W.Workload("fp8q8", 1, 4, 600, 64, "e4m3", False, seed=3)
    q, k, v = W.make_inputs(w)
    o, lse = run_fp8(w, q, k, v, scale=8 * w.scale)
    check_fp8(w, o, lse, q, k, v, scale=8 * w.scale)


@pytest.mark.gpu
@pytest.mark.parametrize("w", [W.N8192_E4M3, W.N8192_E4M3_CAUSAL], ids=lambda w: w.name)
def test_fp8_headline_shape(w):
    q, k, v = W.make_inputs(w)
    o, lse = run_fp8(w, q, k, v)
    check_fp8(w, o, lse, q, k, v, heads=W.sample_heads(w, 2),
              rows=W.sample_rows(w.N, 512))


@pytest.mark.gpu
def test_fp8_long_context_d128():
    # B1 H32 N32768 d128 causal (inputs N(0,1)/2), the shape where e4m3 runs
    # faster than bf16: 2 sampled heads, 256 sampled query rows each
    w = W.LONG_E4M3
    q, k, v = W.make_inputs(w)
    o, lse = run_fp8(w, q, k, v)
    check_fp8(w, o, lse, q, k, v, heads=W.sample_heads(w, 2),
              rows=W.sample_rows(w.N, 256))


# ---------------------------------------------------------------- host side
P = 0x10000


def call8(**kw):
    a = dict(q=P, k=P, v=P, o=P, lse=P, B=1, H=1, Nq=128, Nk=128, d=64, causal=0,
             scale=0.125, qd=1.0, kd=1.0, vd=1.0)
    a.update(kw)
    return b.fa_fwd_fp8_raw(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"],
                            a["Nq"], a["Nk"], a["d"], a["causal"], a["scale"], a["qd"],
                            a["kd"], a["vd"], ctypes.c_void_p(0))


@pytest.mark.parametrize("kw,code", [
    (dict(qd=0.0), b.FA_ERR_SCALE), (dict(kd=-1.0), b.FA_ERR_SCALE),
    (dict(vd=float("nan")), b.FA_ERR_SCALE), (dict(scale=0.0), b.FA_ERR_SCALE),
    (dict(d=32), b.FA_ERR_HEADDIM), (dict(Nk=-3), b.FA_ERR_SHAPE),
    (dict(v=0), b.FA_ERR_NULL), (dict(o=P + 2), b.FA_ERR_ALIGN),
])
def test_fp8_host_checks(kw, code):
    assert call8(**kw) == code


def test_fp8_empty_problem():
    assert call8(q=0, k=0, v=0, o=0, lse=0, Nq=0) == b.FA_OK


def test_fp8_wrapper_rejects_other_dtypes():
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        fa.fwd_fp8(q, q, q, 1.0, 1.0, 1.0)


def test_e4m3_rounding_bound_behind_the_tolerance():
    # The tolerance above rests on |Q(p) - p| <= 2^-4 p + 2^-10 for e4m3
    # round-to-nearest over the range P takes (0 .. 256, within e4m3's 448):
    # 3 mantissa bits give half a unit of 2^-3 relative for normal values,
    # and subnormals are spaced 2^-9 apart.  A dense sweep checks it, and that
    # it is close to tight (a 2^-5 relative bound fails).
    p = torch.cat([torch.linspace(0.0, 256.0, 1_000_001, dtype=torch.float64),
                   torch.linspace(0.0, 0.02, 100_001, dtype=torch.float64)])
    qp = p.float().to(torch.float8_e4m3fn).double()
    err = (qp - p).abs()
    assert bool((err <= 2.0 ** -4 * p + 2.0 ** -10).all())
    assert bool((err > 2.0 ** -5 * p + 2.0 ** -10).any())
    assert float(torch.tensor(256.0).to(torch.float8_e4m3fn).double()) == 256.0
