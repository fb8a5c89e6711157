"""Seeded synthetic inputs and the workload shapes they are drawn for.

This module holds no attention arithmetic: it only names the shapes, draws
the random inputs and counts work.  Both the CUDA path's tests/benchmark and
the oracle's tests take their inputs from here, so the two sides see the
same values.

Shapes follow the pages' forward-time tables (baguaai.com benchmarks page,
"各 GPU 速度对比": batch 8, 32 heads, head dim 64, sequence 512 to 8192;
A10G rows at batch 4) plus a long-context case with 7B-model-shaped heads
(32 heads of dim 128).  Inputs are i.i.d. N(0, 1), drawn in fp32 from a
seeded CPU generator in the order q, k, v, then multiplied by an exact
power of two where a case asks for it, then rounded to nearest into the
storage dtype.
"""
from dataclasses import dataclass, field
import math

import torch

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16,
          "e4m3": torch.float8_e4m3fn}
# Per-tensor descale of the e4m3 inputs: x is stored as round(x / E4M3_DESCALE),
# which keeps N(0, 1) data (|x| < 14) inside e4m3's range (448).
E4M3_DESCALE = 1.0 / 32.0


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str                 # "fp16" | "bf16" | "e4m3"
    causal: bool
    seed: int = 0
    q_mult: float = 1.0        # exact power of two applied to q
    in_mult: float = 1.0       # exact power of two applied to q, k and v
    Nk: int = None             # key length; None means Nk == N

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.d)

    @property
    def n_keys(self):
        return self.N if self.Nk is None else self.Nk

    def flops(self):
        """Counted FLOPs: 4*B*H*Nq*Nk*d, half of it when causal.

        The causal figure is the usual convention (the masked half of the
        diagonal tiles is not subtracted); it is exact for Nq == Nk in the
        limit and is what the throughput metric divides by.
        """
        f = 4.0 * self.B * self.H * self.N * self.n_keys * self.d
        return f / 2.0 if self.causal else f

    def hbm_bytes(self):
        """Algorithmic HBM bytes: read Q, K, V once at their element size,
        write O once (2 B; bf16 for e4m3 inputs) and the fp32 LSE."""
        e = 1 if self.dtype == "e4m3" else 2     # O is bf16 for e4m3 inputs
        bh = self.B * self.H
        return bh * ((self.N + 2 * self.n_keys) * self.d * e
                     + self.N * self.d * 2 + 4 * self.N)

    def kv_bytes(self):
        """Bytes of K and V together (fp16/bf16)."""
        return 2 * self.B * self.H * self.n_keys * self.d * 2

    def with_(self, **kw):
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


# The five configurations (tiny correctness case, N=512 fp16 with a large-
# logit variant, N=2048 bf16, N=8192 bf16 with its sweep, long context).
TINY = Workload("tiny_b1h2n128d64_fp16", 1, 2, 128, 64, "fp16", False, seed=0)
N512 = Workload("b8h32n512d64_fp16", 8, 32, 512, 64, "fp16", False, seed=0)
N512_Q8 = N512.with_(name="b8h32n512d64_fp16_q8", seed=1, q_mult=8.0)
N2048_CAUSAL = Workload("b8h32n2048d64_bf16_causal", 8, 32, 2048, 64, "bf16",
                        True, seed=0)
N2048 = N2048_CAUSAL.with_(name="b8h32n2048d64_bf16", causal=False)
N8192 = Workload("b8h32n8192d64_bf16", 8, 32, 8192, 64, "bf16", False, seed=0)
N8192_CAUSAL = N8192.with_(name="b8h32n8192d64_bf16_causal", causal=True)
LONG = Workload("b1h32n32768d128_bf16_causal", 1, 32, 32768, 128, "bf16",
                True, seed=0, in_mult=0.5)
SWEEP_N = (512, 1024, 2048, 4096, 8192)


N8192_E4M3 = N8192.with_(name="b8h32n8192d64_e4m3", dtype="e4m3")
N8192_E4M3_CAUSAL = N8192_E4M3.with_(name="b8h32n8192d64_e4m3_causal", causal=True)
LONG_E4M3 = LONG.with_(name="b1h32n32768d128_e4m3_causal", dtype="e4m3")


def dequantized(t, dtype):
    """The real values an input tensor stands for, in float64."""
    if dtype == "e4m3":
        return t.double() * E4M3_DESCALE
    return t.double()


def sweep(causal=False):
    return [N8192.with_(name="b8h32n%dd64_bf16%s" % (n, "_causal" if causal else ""),
                        N=n, causal=causal) for n in SWEEP_N]


def make_inputs(w, device="cpu"):
    """Draw q, k, v for workload ``w``: [B, H, N, d] in w.dtype.

    Seeded CPU generator, fp32 N(0,1) in the order q, k, v, exact power-of-
    two multipliers, then round-to-nearest into the dtype.  The values do
    not depend on ``device``; the tensors are moved there after rounding.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(int(w.seed))
    dt = DTYPES[w.dtype]
    shp_q = (w.B, w.H, w.N, w.d)
    shp_k = (w.B, w.H, w.n_keys, w.d)
    q = torch.randn(shp_q, generator=g, dtype=torch.float32)
    k = torch.randn(shp_k, generator=g, dtype=torch.float32)
    v = torch.randn(shp_k, generator=g, dtype=torch.float32)
    if w.q_mult != 1.0:
        q.mul_(w.q_mult)
    if w.in_mult != 1.0:
        q.mul_(w.in_mult)
        k.mul_(w.in_mult)
        v.mul_(w.in_mult)
    if w.dtype == "e4m3":
        # saturating quantisation (e4m3 has no infinity; out of range is NaN)
        out = tuple((t / E4M3_DESCALE).clamp(-448.0, 448.0).to(dt) for t in (q, k, v))
    else:
        out = tuple(t.to(dt) for t in (q, k, v))
    if device != "cpu":
        out = tuple(t.to(device) for t in out)
    return out


def make_inputs_on(w, device):
    """q, k, v of workload ``w`` drawn directly on ``device`` from a seeded
    generator of that device: the same distribution, scaling and rounding as
    ``make_inputs`` (the values differ from the CPU recipe's).  For timing
    runs of shapes whose parity is checked with ``make_inputs`` inputs; it
    saves drawing gigabytes on the host."""
    g = torch.Generator(device=device)
    g.manual_seed(int(w.seed))
    dt = DTYPES[w.dtype]
    shp_q = (w.B, w.H, w.N, w.d)
    shp_k = (w.B, w.H, w.n_keys, w.d)
    out = []
    for shp, mult in ((shp_q, w.q_mult * w.in_mult), (shp_k, w.in_mult), (shp_k, w.in_mult)):
        t = torch.randn(shp, generator=g, dtype=torch.float32, device=device)
        if mult != 1.0:
            t.mul_(mult)
        if w.dtype == "e4m3":
            t = (t / E4M3_DESCALE).clamp_(-448.0, 448.0)
        out.append(t.to(dt))
        del t
    return tuple(out)


def make_upstream_grad(w, seed_offset=1000):
    """dO for the backward: i.i.d. N(0, 1) like q, from its own seed."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(w.seed) + seed_offset)
    t = torch.randn((w.B, w.H, w.N, w.d), generator=g, dtype=torch.float32)
    return t.to(DTYPES[w.dtype])


def sample_heads(w, count, seed=1234):
    """``count`` distinct (b, h) pairs, drawn without replacement."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    perm = torch.randperm(w.B * w.H, generator=g)[:count].tolist()
    return [(i // w.H, i % w.H) for i in perm]


def sample_rows(n, count, seed=1234):
    """``count`` sorted query rows of [0, n), always with 0 and n - 1."""
    if count >= n:
        return list(range(n))
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 1)
    inner = (torch.randperm(n - 2, generator=g)[:count - 2] + 1).tolist()
    return sorted(set([0, n - 1] + inner))
