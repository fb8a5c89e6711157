"""Pins for the fp64 backward oracle (no GPU).

The gradients of L = sum(O * dO) are pinned to what the mathematics fixes:
hand-derived worked examples, central finite differences of the (separately pinned) forward oracle along
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


# ---------------------------------------------------------------- worked examples
def test_two_key_worked_example():
    # d = 2, scale 1/2, one query q = (2a, 2 ln 3), keys k0 = (1, 0),
    # k1 = (1, 1): logits (a, a + ln 3), so p = (1/4, 3/4).  v0 = (4, 0),
    # v1 = (0, 8) give O = (1, 6).  Upstream g = (1, 2):
    #   D = g.O = 13,  dP = (g.v0, g.v1) = (4, 16),
    #   dS = p * (dP - D) = (-9/4, 9/4),
    #   dV_j = p_j g = (1/4, 1/2), (3/4, 3/2),
    #   dQ = scale * sum_j dS_j k_j = (0, 9/8),
    #   dK_j = scale * dS_j q = dS_j * (a, ln 3).
    # A dropped scale doubles dQ and dK; a flipped sign or a transposed K
    # changes every entry.
    a, ln3 = 0.5, np.log(3.0)
    q = np.array([[2 * a, 2 * ln3]])
    k = np.array([[1.0, 0.0], [1.0, 1.0]])
    v = np.array([[4.0, 0.0], [0.0, 8.0]])
    g = np.array([[1.0, 2.0]])
    dq, dk, dv = oracle.attention_bwd(q, k, v, g, 0.5, False)
    np.testing.assert_allclose(dq, [[0.0, 9 / 8]], rtol=0, atol=1e-14)
    np.testing.assert_allclose(dk, [[-9 / 4 * a, -9 / 4 * ln3], [9 / 4 * a, 9 / 4 * ln3]],
                               rtol=0, atol=1e-14)
    np.testing.assert_allclose(dv, [[0.25, 0.5], [0.75, 1.5]], rtol=0, atol=1e-14)


def test_causal_worked_example():
    # d = 1, scale 1, q = (1, 1), k = (0, ln 3), v = (2, 6), g = (1, 1).
    # Row 0 sees key 0 only: p = (1, 0), O = 2, dS = 1 * (2 - 2) = 0.
    # Row 1 sees both: p = (1/4, 3/4), O = 5, dP = (2, 6),
    #   dS = (1/4 (2 - 5), 3/4 (6 - 5)) = (-3/4, 3/4), dQ_1 = 3/4 ln 3.
    # Summed over rows: dV = (1 + 1/4, 3/4), dK = (-3/4, 3/4).  With the mask
    # reversed, row 0 would see key 1 and every entry would change.
    ln3 = np.log(3.0)
    q = np.array([[1.0], [1.0]])
    k = np.array([[0.0], [ln3]])
    v = np.array([[2.0], [6.0]])
    g = np.array([[1.0], [1.0]])
    dq, dk, dv = oracle.attention_bwd(q, k, v, g, 1.0, True)
    np.testing.assert_allclose(dq, [[0.0], [0.75 * ln3]], rtol=0, atol=1e-14)
    np.testing.assert_allclose(dk, [[-0.75], [0.75]], rtol=0, atol=1e-14)
    np.testing.assert_allclose(dv, [[1.25], [0.75]], rtol=0, atol=1e-14)


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
