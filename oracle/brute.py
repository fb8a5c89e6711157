"""Unfused brute-force attention in pure Python (tiny shapes only).

TEST INFRASTRUCTURE ONLY: the product path never imports this module.

This is the "standard" attention that the pages contrast with the fused
kernel: it materialises the whole score matrix and the whole probability
matrix before the weighted sum (zzycbzc.com/news/393333, section
"技术痛点"; baguaai.com benchmarks page, the "标准" columns and the
"注意力矩阵" column of the memory table).  It is structured differently
from the C oracle on purpose (full matrices, probabilities normalised
before the product, exactly rounded sums via math.fsum) so that the two
check each other.
"""
import math

NEG_INF = float("-inf")


def attention_brute(q, k, v, scale, causal):
    """q: Nq x d, k, v: Nk x d nested lists of floats (one head).

    Returns (O as Nq x d lists, LSE as a list of Nq floats, P as Nq x Nk).
    Causal allows key j for query i iff j <= i + (Nk - Nq).
    """
    nq, nk = len(q), len(k)
    d = len(q[0]) if nq else 0
    # full score matrix, masked entries -inf
    s = [[NEG_INF] * nk for _ in range(nq)]
    for i in range(nq):
        for j in range(nk):
            if causal and j > i + (nk - nq):
                continue
            s[i][j] = scale * math.fsum(q[i][t] * k[j][t] for t in range(d))
    # full probability matrix, one row at a time
    p = [[0.0] * nk for _ in range(nq)]
    lse = [NEG_INF] * nq
    for i in range(nq):
        finite = [x for x in s[i] if x != NEG_INF]
        if not finite:
            continue
        mx = max(finite)
        e = [math.exp(x - mx) if x != NEG_INF else 0.0 for x in s[i]]
        tot = math.fsum(e)
        p[i] = [x / tot for x in e]
        lse[i] = mx + math.log(tot)
    # O = P V
    o = [[math.fsum(p[i][j] * v[j][t] for j in range(nk)) for t in range(d)]
         for i in range(nq)]
    return o, lse, p


def attention_brute_bwd(q, k, v, dout, scale, causal):
    """Unfused backward (tiny shapes): full P, dP and dS matrices.
    Returns dQ, dK, dV as nested lists."""
    o, _, p = attention_brute(q, k, v, scale, causal)
    nq, nk = len(q), len(k)
    d = len(q[0]) if nq else 0
    dv = [[math.fsum(p[i][j] * dout[i][t] for i in range(nq)) for t in range(d)]
          for j in range(nk)]
    dp = [[math.fsum(dout[i][t] * v[j][t] for t in range(d)) for j in range(nk)]
          for i in range(nq)]
    dd = [math.fsum(dout[i][t] * o[i][t] for t in range(d)) for i in range(nq)]
    ds = [[p[i][j] * (dp[i][j] - dd[i]) for j in range(nk)] for i in range(nq)]
    dq = [[scale * math.fsum(ds[i][j] * k[j][t] for j in range(nk)) for t in range(d)]
          for i in range(nq)]
    dk = [[scale * math.fsum(ds[i][j] * q[i][t] for i in range(nq)) for t in range(d)]
          for j in range(nk)]
    return dq, dk, dv
