"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded, rounded inputs.

Tolerances (O compared in fp64 against the unrounded oracle O; max and mean
of |dO| over every compared element):
    fp16 inputs: max <= 5e-3, mean <= 5e-4
    bf16 inputs: max <= 2e-2, mean <= 2e-3
    LSE (fp32):  max |dLSE| <= 1e-3
Full-size workloads run on the GPU exactly as the benchmark launches them;
the oracle then checks sampled (batch, head) slices, and sampled rows for
the long-context case.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_39_gb300 as fa
from exact_attention_39_gb300 import workloads as W
import oracle

pytestmark = pytest.mark.gpu

TOL = {"fp16": (5e-3, 5e-4), "bf16": (2e-2, 2e-3)}
LSE_TOL = 1e-3


def run_gpu(w, q, k, v):
    dev = torch.device("cuda")
    o, lse = fa.fwd(q.to(dev), k.to(dev), v.to(dev), causal=w.causal,
                    scale=w.scale)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    return o.cpu(), lse.cpu()


def as64(t):
    return t.double().numpy()


def check(w, o_gpu, lse_gpu, q, k, v, heads=None, rows=None):
    """Compare GPU outputs with the oracle on the (b, h) pairs ``heads``
    (all when None) and query ``rows`` (all when None)."""
    if heads is None:
        qs, ks, vs = as64(q), as64(k), as64(v)
        og, lg = as64(o_gpu), as64(lse_gpu)
    else:
        idx = torch.tensor([b * w.H + h for b, h in heads])
        flat = lambda t: t.reshape(w.B * w.H, *t.shape[2:])[idx]
        qs, ks, vs = as64(flat(q)), as64(flat(k)), as64(flat(v))
        og, lg = as64(flat(o_gpu)), as64(flat(lse_gpu))
    if rows is not None:
        og, lg = og[..., rows, :], lg[..., rows]
    o_ref, lse_ref = oracle.attention_fwd(qs, ks, vs, w.scale, w.causal, rows=rows)
    assert np.isfinite(og).all() and np.isfinite(lg).all()
    d_o = np.abs(og - o_ref)
    d_l = np.abs(lg - lse_ref)
    mx, mean = TOL[w.dtype]
    msg = "%s: max|dO|=%.3g mean|dO|=%.3g max|dLSE|=%.3g" % (
        w.name, d_o.max(), d_o.mean(), d_l.max())
    assert d_o.max() <= mx and d_o.mean() <= mean and d_l.max() <= LSE_TOL, msg
    return d_o.max(), d_o.mean(), d_l.max()


def full_check(w):
    q, k, v = W.make_inputs(w)
    o, lse = run_gpu(w, q, k, v)
    return check(w, o, lse, q, k, v)


# ------------------------------------------------------------ the five configs
def test_config_tiny():
    full_check(W.TINY)


@pytest.mark.parametrize("w", [W.N512, W.N512_Q8], ids=lambda w: w.name)
def test_config_n512_fp16(w):
    full_check(w)


@pytest.mark.parametrize("w", [W.N2048_CAUSAL, W.N2048], ids=lambda w: w.name)
def test_config_n2048_bf16(w):
    q, k, v = W.make_inputs(w)
    o, lse = run_gpu(w, q, k, v)
    check(w, o, lse, q, k, v, heads=W.sample_heads(w, 16))


@pytest.mark.parametrize("w", [W.N8192, W.N8192_CAUSAL], ids=lambda w: w.name)
def test_config_n8192_bf16(w):
    q, k, v = W.make_inputs(w)
    o, lse = run_gpu(w, q, k, v)
    check(w, o, lse, q, k, v, heads=W.sample_heads(w, 4))


def test_config_long_context_d128():
    w = W.LONG
    q, k, v = W.make_inputs(w)
    o, lse = run_gpu(w, q, k, v)
    check(w, o, lse, q, k, v, heads=W.sample_heads(w, 2),
          rows=W.sample_rows(w.N, 256))


@pytest.mark.parametrize("n", [512, 1024, 4096])
@pytest.mark.parametrize("causal", [False, True])
def test_sequence_sweep(n, causal):
    w = W.N8192.with_(name="sweep%d" % n, N=n, causal=causal)
    q, k, v = W.make_inputs(w)
    o, lse = run_gpu(w, q, k, v)
    check(w, o, lse, q, k, v, heads=W.sample_heads(w, 2))


# ------------------------------------------------------------ ragged and small
# 16-bit inputs at d = 64 with at most 4096 keys run one query tile per CTA,
# K and V on separate ring barriers; 640 and 1000 keys wrap the two-stage
# ring several times.
@pytest.mark.parametrize("n", [1, 2, 3, 64, 127, 128, 129, 255, 256, 257, 300, 511, 512, 513,
                               640, 1000])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_lengths_d64(n, causal):
    for dtype in ("fp16", "bf16"):
        w = W.Workload("ragged", 1, 3, n, 64, dtype, causal, seed=n)
        full_check(w)


# Above 4096 keys 16-bit inputs at d = 64 run two query tiles per CTA.  Short
# query lengths against 4095..5000 keys straddle the switch and reach the
# two-tile kernel with ragged query and key tails at sizes the oracle
# finishes quickly.
@pytest.mark.parametrize("nq,nk", [(300, 4095), (300, 4096), (300, 4097), (1, 4353),
                                   (127, 4200), (129, 4200), (256, 4224), (257, 4500),
                                   (511, 4097), (513, 5000), (1000, 4300)])
@pytest.mark.parametrize("causal", [False, True])
def test_shape_switch_and_two_tile_d64(nq, nk, causal):
    for dtype in ("fp16", "bf16"):
        w = W.Workload("two_tile", 1, 2, nq, 64, dtype, causal, seed=nq + 3 * nk, Nk=nk)
        full_check(w)


# Causal problems with more than 4096 keys run the two-tile shape in which the
# first tile skips a key block wholly past its diagonal; ragged lengths and
# Nq != Nk move that block's position and the first tile's block count.
@pytest.mark.parametrize("nq,nk", [(4097, 4097), (4200, 4200), (4353, 4353), (4500, 4500),
                                   (5119, 5119), (4300, 4500), (4500, 4300), (700, 4200),
                                   (4400, 4300), (260, 4353)])
def test_causal_tile_skip_lengths(nq, nk):
    for dtype in ("fp16", "bf16"):
        w = W.Workload("skip", 1, 3, nq, 64, dtype, True, seed=nq + 7 * nk, Nk=nk)
        q, k, v = W.make_inputs(w)
        o, lse = run_gpu(w, q, k, v)
        n_dead = max(0, nq - nk)
        if n_dead:
            assert (o[:, :, :n_dead] == 0).all()
            assert torch.isinf(lse[:, :, :n_dead]).all()
        check(w, o, lse, q, k, v, rows=list(range(n_dead, nq)))


@pytest.mark.parametrize("n", [1, 100, 128, 256, 383, 512, 777])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_lengths_d128(n, causal):
    for dtype in ("fp16", "bf16"):
        w = W.Workload("ragged128", 2, 2, n, 128, dtype, causal, seed=n + 1)
        full_check(w)


@pytest.mark.parametrize("nq,nk", [(1, 1000), (64, 777), (300, 128), (128, 300),
                                   (1000, 257), (257, 1000), (513, 2048), (2048, 100)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_query_and_key_lengths_differ(nq, nk, causal, d):
    # bottom-right causal alignment; rows that see no key give O = 0, LSE = -inf
    w = W.Workload("qk", 1, 2, nq, d, "bf16" if d == 64 else "fp16", causal,
                   seed=nq + nk, Nk=nk)
    q, k, v = W.make_inputs(w)
    o, lse = run_gpu(w, q, k, v)
    n_dead = max(0, nq - nk) if causal else 0
    if n_dead:
        assert (o[:, :, :n_dead] == 0).all()
        assert torch.isinf(lse[:, :, :n_dead]).all() and (lse[:, :, :n_dead] < 0).all()
    live = list(range(n_dead, nq))
    check(w, o, lse, q, k, v, rows=live)


def test_no_keys_at_all():
    w = W.Workload("nokeys", 2, 2, 200, 64, "bf16", False, seed=9, Nk=0)
    q = W.make_inputs(w.with_(Nk=None))[0].cuda()
    kv = torch.empty(2, 2, 0, 64, dtype=q.dtype, device="cuda")
    o, lse = fa.fwd(q, kv, kv)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    assert (o == 0).all() and torch.isinf(lse).all() and (lse < 0).all()


def test_large_logits_d128():
    w = W.Workload("q8_d128", 1, 4, 700, 128, "fp16", False, seed=5, q_mult=8.0)
    full_check(w)
    full_check(w.with_(causal=True))


# ------------------------------------------------------------ closed forms on the GPU
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_is_mean_of_values(d, causal):
    n = 400
    w = W.Workload("zeroq", 1, 2, n, d, "bf16", causal, seed=3)
    q, k, v = W.make_inputs(w)
    q = torch.zeros_like(q)
    o, lse = run_gpu(w, q, k, v)
    vd = v.double()
    cnt = torch.arange(1, n + 1, dtype=torch.float64) if causal else torch.full((n,), float(n), dtype=torch.float64)
    mean = vd.cumsum(2) / cnt[:, None] if causal else vd.mean(2, keepdim=True).expand_as(vd)
    assert (o.double() - mean).abs().max() <= 2e-2
    assert (lse.double() - cnt.log()).abs().max() <= 1e-3


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_constant_values(dtype):
    w = W.Workload("constv", 2, 2, 333, 64, dtype, True, seed=4)
    q, k, v = W.make_inputs(w)
    row = torch.linspace(-3, 3, 64).to(W.DTYPES[dtype])
    v = row.expand_as(v).contiguous()
    o, _ = run_gpu(w, q, k, v)
    # Every softmax row sums to one, so O reproduces the constant row.  The
    # kernel rounds each p_j to the dtype (relative error <= u, the unit
    # roundoff: 2^-8 bf16, 2^-11 fp16) while l sums the unrounded p_j, so
    # O = v * sum(round(p_j)) / sum(p_j) is within u * |v| of v; then O is
    # rounded to the dtype once more (half an ulp of |v| (1 + u)).  bf16:
    # 3 * 2^-8 + 2^-7 = 1.95e-2; fp16: 3 * 2^-11 + 2^-10 = 2.44e-3.
    u = {"bf16": 2.0 ** -8, "fp16": 2.0 ** -11}[dtype]
    vmax = 3.0
    half_ulp = 2.0 ** (math.floor(math.log2(vmax * (1 + u)))) * u
    bound = vmax * u + half_ulp + 1e-6          # + fp32 accumulation
    assert bound <= TOL[dtype][0]
    assert (o.double() - row.double()).abs().max() <= bound


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_standard_comparator_computes_attention(causal, dtype):
    # The unfused "standard" attention the benchmark times against fa_fwd
    # (S materialised in the dtype, fp32 softmax, torch/cuBLAS on the GPU)
    # computes the same attention: O against the oracle at the dtype's
    # tolerance, on B1 H2 N256 d64.
    import bench
    w = W.Workload("standard", 1, 2, 256, 64, dtype, causal, seed=12)
    q, k, v = W.make_inputs(w)
    o = bench.standard_attention(q.cuda(), k.cuda(), v.cuda(), causal, w.scale)
    torch.cuda.synchronize()
    o_ref, _ = oracle.attention_fwd(as64(q), as64(k), as64(v), w.scale, causal)
    d_o = np.abs(as64(o.cpu()) - o_ref)
    mx, mean = TOL[dtype]
    assert d_o.max() <= mx and d_o.mean() <= mean, (d_o.max(), d_o.mean())


def test_single_key_and_causal_first_row():
    w = W.Workload("first", 1, 2, 1, 64, "fp16", False, seed=6)
    q, k, v = W.make_inputs(w)
    o, lse = run_gpu(w, q, k, v)
    assert torch.equal(o, v)          # one key: O = v0 exactly
    dot = (q.double() * k.double()).sum(-1) * w.scale
    assert (lse.double() - dot).abs().max() <= 1e-3
    w = W.Workload("first", 1, 2, 500, 64, "fp16", True, seed=6)
    q, k, v = W.make_inputs(w)
    o, _ = run_gpu(w, q, k, v)
    assert torch.equal(o[:, :, 0], v[:, :, 0])   # causal row 0 sees key 0 only


# ------------------------------------------------------------ launch behaviour
def test_deterministic_and_stream_ordered():
    w = W.N2048_CAUSAL.with_(B=2)
    q, k, v = (t.cuda() for t in W.make_inputs(w))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())   # the inputs' copies come first
    with torch.cuda.stream(s):
        o1, l1 = fa.fwd(q, k, v, causal=True, stream=s)
        o2, l2 = fa.fwd(q, k, v, causal=True, stream=s)
    s.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert fa.last_device_error(s) == 0


def test_host_buffers_end_to_end():
    w = W.N512.with_(B=2, H=4)
    q, k, v = W.make_inputs(w)
    pin = lambda t: t.pin_memory()
    qh, kh, vh = pin(q), pin(k), pin(v)
    dev = [torch.empty_like(t, device="cuda") for t in (q, k, v)]
    od = torch.empty_like(dev[0])
    ld = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device="cuda")
    oh = torch.empty_like(q).pin_memory()
    lh = torch.empty(w.B, w.H, w.N, dtype=torch.float32).pin_memory()
    fa.fwd_host(qh, kh, vh, *dev, od, ld, oh, lh, causal=False, scale=w.scale)
    check(w, oh, lh, q, k, v)


@pytest.mark.parametrize("B,H,N,causal,dtype", [
    (1, 1, 200, False, "fp16"), (1, 5, 384, True, "bf16"),
    (3, 7, 300, True, "bf16"), (2, 16, 1024, False, "bf16")])
def test_host_buffers_match_device_call(B, H, N, causal, dtype):
    # The chunked host-buffer pipeline runs the same kernel per (batch, head)
    # problem, so its outputs equal the device-buffer call bit for bit, for
    # head counts that do and do not divide into the chunks.
    w = W.Workload("host", B, H, N, 64, dtype, causal, seed=21)
    q, k, v = W.make_inputs(w)
    qh, kh, vh = (t.pin_memory() for t in (q, k, v))
    dev = [torch.empty_like(t, device="cuda") for t in (q, k, v)]
    od = torch.empty_like(dev[0])
    ld = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
    oh = torch.empty_like(q).pin_memory()
    lh = torch.empty(B, H, N, dtype=torch.float32).pin_memory()
    fa.fwd_host(qh, kh, vh, *dev, od, ld, oh, lh, causal=causal, scale=w.scale)
    o_ref, l_ref = fa.fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal,
                          scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(oh, o_ref.cpu()) and torch.equal(lh, l_ref.cpu())
    assert fa.last_device_error() == 0


def test_wrappers_reject_buffers_off_the_device():
    # Every pointer the library receives is dereferenced on the current
    # device, so the wrappers refuse host or non-contiguous tensors before
    # anything is enqueued.
    w = W.Workload("dev", 1, 2, 128, 64, "bf16", False, seed=3)
    q, k, v = (t.cuda() for t in W.make_inputs(w))
    lse = torch.empty(1, 2, 128, dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        fa.fwd(q, k, v, out=torch.empty_like(q, device="cpu"))
    with pytest.raises(ValueError):
        fa.fwd(q, k, v, lse=lse.cpu())
    with pytest.raises(ValueError):
        fa.fwd(q, k, v, out=torch.empty(1, 2, 64, 128, dtype=q.dtype,
                                        device="cuda").transpose(2, 3))
    with pytest.raises(ValueError):
        fa.fwd(q, k.cpu(), v)
    o, lse = fa.fwd(q, k, v)
    with pytest.raises(ValueError):
        fa.bwd(q, k, v, o, lse, o, workspace=torch.empty(1 << 12, dtype=torch.uint8))
    with pytest.raises(ValueError):
        fa.bwd(q, k, v, o, lse, o, dq=torch.empty_like(q, device="cpu"))
    q8 = q.to(torch.float8_e4m3fn)
    with pytest.raises(ValueError):
        fa.fwd_fp8(q8, q8, q8, 1.0, 1.0, 1.0, lse=lse.cpu())
    host = [t.cpu().pin_memory() for t in (q, k, v)]
    oh = torch.empty_like(host[0]).pin_memory()
    lh = torch.empty(1, 2, 128, dtype=torch.float32).pin_memory()
    with pytest.raises(ValueError):
        fa.fwd_host(*host, q, k, v.cpu(), o, lse, oh, lh)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0


def test_outputs_do_not_touch_neighbours():
    # O and LSE are written only inside their [B, H, N, d] / [B, H, N] spans.
    w = W.Workload("guard", 1, 2, 300, 64, "bf16", True, seed=8)
    q, k, v = (t.cuda() for t in W.make_inputs(w))
    n_o = q.numel()
    buf = torch.full((n_o + 2048,), 7.0, dtype=q.dtype, device="cuda")
    lbuf = torch.full((w.B * w.H * w.N + 256,), 7.0, dtype=torch.float32, device="cuda")
    o = buf[1024:1024 + n_o].view_as(q)
    lse = lbuf[128:128 + w.B * w.H * w.N].view(w.B, w.H, w.N)
    fa.fwd(q, k, v, causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    assert (buf[:1024] == 7).all() and (buf[1024 + n_o:] == 7).all()
    assert (lbuf[:128] == 7).all() and (lbuf[128 + w.B * w.H * w.N:] == 7).all()
