"""Pins for the fp64 backward oracle (no GPU).

The gradients of L = sum(O * dO) are pinned to what the mathematics fixes:
central finite differences of the (separately pinned) forward oracle along
random directions, an unfused brute force, closed forms and invariants of
the softmax Jacobian.
"""
import numpy as np
import pytest

import oracle
from oracle.brute import attention_brute_bwd


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def loss(q, k, v, g, scale, causal):
    o, _ = oracle.attention_fwd(q, k, v, scale, causal)
    return float(np.sum(o * g))


@pytest.mark.parametrize("nq,nk,causal", [(24, 24, False), (24, 24, True),
                                          (10, 30, True), (30, 10, True), (17, 9, False)])
def test_gradients_match_finite_differences(nq, nk, causal):
    d, scale, eps = 8, 0.4, 1e-5
    q, k, v = rnd((nq, d), 1), rnd((nk, d), 2), rnd((nk, d), 3)
    g = rnd((nq, d), 4)
    dq, dk, dv = oracle.attention_bwd(q, k, v, g, scale, causal)
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for seed in (10, 11):
            u = rnd(x.shape, seed)
            args = {"q": q, "k": k, "v": v}
            args[name] = x + eps * u
            lp = loss(args["q"], args["k"], args["v"], g, scale, causal)
            args[name] = x - eps * u
            lm = loss(args["q"], args["k"], args["v"], g, scale, causal)
            num = (lp - lm) / (2 * eps)
            ana = float(np.sum(grad * u))
            assert abs(num - ana) <= 1e-7 * max(1.0, abs(ana)), (name, num, ana)


@pytest.mark.parametrize("nq,nk,causal", [(7, 7, True), (5, 9, True), (9, 5, False), (1, 4, True)])
def test_agrees_with_brute_force(nq, nk, causal):
    d, scale = 4, 0.5
    q, k, v, g = rnd((nq, d), 5), rnd((nk, d), 6), rnd((nk, d), 7), rnd((nq, d), 8)
    dq, dk, dv = oracle.attention_bwd(q, k, v, g, scale, causal)
    bq, bk, bv = attention_brute_bwd(q.tolist(), k.tolist(), v.tolist(), g.tolist(),
                                     scale, causal)
    np.testing.assert_allclose(dq, bq, atol=1e-12)
    np.testing.assert_allclose(dk, bk, atol=1e-12)
    np.testing.assert_allclose(dv, bv, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_softmax_jacobian_identities(causal):
    n, d, scale = 40, 16, 0.25
    q, k, v, g = rnd((n, d), 9), rnd((n, d), 10), rnd((n, d), 11), rnd((n, d), 12)
    dq, dk, dv = oracle.attention_bwd(q, k, v, g, scale, causal)
    # every row of P sums to one: the dV rows add up to the dO rows
    np.testing.assert_allclose(dv.sum(axis=0), g.sum(axis=0), atol=1e-12)
    # every row of dS sums to zero: so do the dK rows
    np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-12)


def test_constant_values_and_zero_upstream():
    n, d = 20, 8
    q, k, g = rnd((n, d), 13), rnd((n, d), 14), rnd((n, d), 15)
    v = np.tile(rnd((d,), 16), (n, 1))
    dq, dk, dv = oracle.attention_bwd(q, k, v, g, 0.5, True)
    np.testing.assert_allclose(dq, 0.0, atol=1e-13)      # O does not depend on Q, K
    np.testing.assert_allclose(dk, 0.0, atol=1e-13)
    dq, dk, dv = oracle.attention_bwd(q, k, rnd((n, d), 17), np.zeros((n, d)), 0.5, False)
    assert not dq.any() and not dk.any() and not dv.any()


def test_key_shift_leaves_query_gradient():
    # O(Q, K + u) = O(Q, K) for every Q, so dQ (and dV) do not change
    n, d = 30, 8
    q, k, v, g = rnd((n, d), 18), rnd((n, d), 19), rnd((n, d), 20), rnd((n, d), 21)
    u = rnd((d,), 22) * 2
    a = oracle.attention_bwd(q, k, v, g, 0.3, True)
    b = oracle.attention_bwd(q, k + u, v, g, 0.3, True)
    np.testing.assert_allclose(a[0], b[0], atol=1e-11)
    np.testing.assert_allclose(a[2], b[2], atol=1e-11)


def test_batched_and_threads():
    B, H, n, d = 2, 2, 33, 8
    q, k, v, g = (rnd((B, H, n, d), s) for s in (23, 24, 25, 26))
    full = oracle.attention_bwd(q, k, v, g, 0.3, True, nthreads=3)
    one = oracle.attention_bwd(q[1, 0], k[1, 0], v[1, 0], g[1, 0], 0.3, True, nthreads=1)
    for a, b in zip(full, one):
        np.testing.assert_allclose(a[1, 0], b, atol=1e-13)
