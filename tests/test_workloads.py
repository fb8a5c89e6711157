"""The seeded input recipe both sides use (no GPU): deterministic, drawn in
the order q, k, v from one generator, exact power-of-two multipliers, then
rounded to nearest into the storage type; e4m3 saturates instead of
overflowing."""
import math

import torch

from exact_attention_39_gb300 import workloads as W


def test_same_seed_same_tensors_and_order():
    w = W.Workload("t", 1, 2, 40, 64, "fp16", False, seed=7)
    a = W.make_inputs(w)
    b = W.make_inputs(w)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    g = torch.Generator(device="cpu")
    g.manual_seed(7)
    ref = [torch.randn((1, 2, 40, 64), generator=g, dtype=torch.float32) for _ in range(3)]
    for x, r in zip(a, ref):                    # q, k, v in that order
        assert torch.equal(x, r.to(torch.float16))


def test_multipliers_are_exact_powers_of_two():
    base = W.Workload("t", 1, 1, 32, 64, "bf16", False, seed=3)
    q0, k0, v0 = W.make_inputs(base)
    q8, k8, _ = W.make_inputs(base.with_(q_mult=8.0))
    assert torch.equal(q8.float(), q0.float() * 8) and torch.equal(k8, k0)
    qh, kh, vh = W.make_inputs(base.with_(in_mult=0.5))
    for x, y in ((qh, q0), (kh, k0), (vh, v0)):
        assert torch.equal(x.float(), y.float() * 0.5)


def test_e4m3_inputs_saturate_and_dequantize():
    w = W.Workload("t", 1, 1, 64, 64, "e4m3", False, seed=5, q_mult=64.0)
    q, k, v = W.make_inputs(w)
    assert q.dtype == torch.float8_e4m3fn
    for t in (q, k, v):
        f = t.float()
        assert torch.isfinite(f).all() and f.abs().max() <= 448.0
    # the real values are the stored ones times the descale
    assert torch.equal(W.dequantized(k, "e4m3"), k.double() * W.E4M3_DESCALE)


def test_counted_work():
    w = W.N8192
    assert w.flops() == 4.0 * 8 * 32 * 8192 * 8192 * 64
    assert W.N8192_CAUSAL.flops() == w.flops() / 2
    assert w.hbm_bytes() == 8 * 32 * (8 * 8192 * 64 + 4 * 8192)
    assert math.isclose(w.scale, 0.125)
    q = W.N8192.with_(Nk=1024)
    assert q.flops() == 4.0 * 8 * 32 * 8192 * 1024 * 64
