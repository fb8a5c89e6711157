"""Pins for the fp64 CPU oracle (no GPU).

The pages print no worked example of the attention values themselves, so the
oracle is pinned by what the mathematics fixes: hand-derived worked
examples, closed forms, invariants, a library routine on the cases that
reduce to one, and an unfused brute force.  Each is chosen so that a
plausible slip in the oracle (a dropped scale, a transposed operand, a wrong
mask direction, a missing max shift, a wrong log base) fails at least one.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle.brute import attention_brute
from exact_attention_39_gb300 import workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# ---------------------------------------------------------------- worked examples
def test_two_key_worked_example():
    # d = 2, one query, keys k0 = (1, 0), k1 = (1, 1); q = (a, ln 3) gives
    # logits s0 = a, s1 = a + ln 3, so p = (1/4, 3/4).  With v0 = (4, 0),
    # v1 = (0, 8): O = (1, 6) and LSE = a + ln 4.  A transposed K would give
    # logits (a + ln3, ln3) instead and fail.
    a = 0.5
    for scale in (1.0, 0.5):
        q = np.array([[a, math.log(3.0)]]) / scale
        k = np.array([[1.0, 0.0], [1.0, 1.0]])
        v = np.array([[4.0, 0.0], [0.0, 8.0]])
        o, lse = oracle.attention_fwd(q, k, v, scale, causal=False)
        np.testing.assert_allclose(o, [[1.0, 6.0]], rtol=0, atol=1e-14)
        assert abs(lse[0] - (a + math.log(4.0))) < 1e-14


def test_causal_worked_example():
    # d = 1, q_i = 1, k = (0, ln 2, ln 3): unnormalised weights 1, 2, 3.
    # v = (6, 12, 18).  Causal rows: O0 = 6, O1 = (6 + 24)/3 = 10,
    # O2 = (6 + 24 + 54)/6 = 14; LSE = (0, ln 3, ln 6).
    q = np.ones((3, 1))
    k = np.array([[0.0], [math.log(2.0)], [math.log(3.0)]])
    v = np.array([[6.0], [12.0], [18.0]])
    o, lse = oracle.attention_fwd(q, k, v, 1.0, causal=True)
    np.testing.assert_allclose(o[:, 0], [6.0, 10.0, 14.0], rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, [0.0, math.log(3), math.log(6)], atol=1e-14)
    # non-causal: every row sees all three keys
    o, lse = oracle.attention_fwd(q, k, v, 1.0, causal=False)
    np.testing.assert_allclose(o[:, 0], [14.0] * 3, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, [math.log(6)] * 3, atol=1e-14)
    # two queries, three keys: the causal mask is aligned to the bottom-right
    # corner, so query i sees keys j <= i + 1.
    o, lse = oracle.attention_fwd(q[:2], k, v, 1.0, causal=True)
    np.testing.assert_allclose(o[:, 0], [10.0, 14.0], rtol=0, atol=1e-13)


def test_fully_masked_row_contract():
    # three queries, one key, causal bottom-right: row 0 and 1 see nothing.
    q = np.ones((3, 2))
    k = np.ones((1, 2))
    v = np.full((1, 2), 7.0)
    o, lse = oracle.attention_fwd(q, k, v, 1.0, causal=True)
    np.testing.assert_array_equal(o[:2], 0.0)
    assert lse[0] == -math.inf and lse[1] == -math.inf
    np.testing.assert_allclose(o[2], [7.0, 7.0])
    assert abs(lse[2] - 2.0) < 1e-15


# ---------------------------------------------------------------- closed forms
@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_gives_mean_of_values(causal):
    n, d = 37, 8
    q = np.zeros((n, d))
    k, v = rnd((n, d), 1), rnd((n, d), 2)
    o, lse = oracle.attention_fwd(q, k, v, 0.125, causal)
    for i in range(n):
        cnt = i + 1 if causal else n
        np.testing.assert_allclose(o[i], v[:cnt].mean(axis=0), atol=1e-13)
        assert abs(lse[i] - math.log(cnt)) < 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_constant_values(causal):
    n, d = 29, 16
    q, k = rnd((n, d), 3), rnd((n, d), 4)
    c = rnd((d,), 5)
    v = np.tile(c, (n, 1))
    o, _ = oracle.attention_fwd(q, k, v, 0.25, causal)
    np.testing.assert_allclose(o, np.tile(c, (n, 1)), atol=1e-13)


def test_single_key():
    d = 8
    q, k, v = rnd((1, d), 6), rnd((1, d), 7), rnd((1, d), 8)
    for causal in (False, True):
        o, lse = oracle.attention_fwd(q, k, v, 0.3, causal)
        np.testing.assert_array_equal(o[0], v[0])
        dot = math.fsum(float(x) * float(y) for x, y in zip(q[0], k[0]))
        assert abs(lse[0] - 0.3 * dot) < 1e-14


def test_causal_first_and_last_rows():
    n, d = 50, 8
    q, k, v = rnd((n, d), 9), rnd((n, d), 10), rnd((n, d), 11)
    oc, lc = oracle.attention_fwd(q, k, v, 0.4, causal=True)
    on, ln_ = oracle.attention_fwd(q, k, v, 0.4, causal=False)
    np.testing.assert_array_equal(oc[0], v[0])
    np.testing.assert_allclose(oc[-1], on[-1], atol=1e-15)
    assert abs(lc[-1] - ln_[-1]) < 1e-15
    # any earlier row must differ (the mask hides keys it would see)
    assert np.abs(oc[n // 2] - on[n // 2]).max() > 1e-3


def test_dominant_key():
    n, d = 20, 4
    q = np.zeros((1, d)); q[0, 0] = 1.0
    k = np.zeros((n, d)); k[13, 0] = 80.0
    v = rnd((n, d), 12)
    o, lse = oracle.attention_fwd(q, k, v, 1.0, causal=False)
    np.testing.assert_allclose(o[0], v[13], atol=1e-15)
    assert abs(lse[0] - 80.0) < 1e-12


def test_large_logits_stay_finite():
    n, d = 64, 16
    q, k, v = rnd((n, d), 13) * 1e3, rnd((n, d), 14), rnd((n, d), 15)
    o, lse = oracle.attention_fwd(q, k, v, 1.0, causal=False)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    s = q @ k.T
    arg = s.argmax(axis=1)
    top2 = np.sort(s, axis=1)[:, -2:]
    clear = (top2[:, 1] - top2[:, 0]) > 60.0    # runner-up weight < e^-60
    assert clear.sum() > n // 2
    np.testing.assert_allclose(o[clear], v[arg][clear], atol=1e-12)


# ---------------------------------------------------------------- invariants
def test_joint_key_value_permutation():
    n, d = 40, 8
    q, k, v = rnd((n, d), 16), rnd((n, d), 17), rnd((n, d), 18)
    perm = np.random.default_rng(19).permutation(n)
    o1, l1 = oracle.attention_fwd(q, k, v, 0.35, causal=False)
    o2, l2 = oracle.attention_fwd(q, k[perm], v[perm], 0.35, causal=False)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)
    # permuting the values alone must change the result
    o3, _ = oracle.attention_fwd(q, k, v[perm], 0.35, causal=False)
    assert np.abs(o3 - o1).max() > 1e-3


def test_row_shift_of_logits():
    # k_j -> k_j + u adds scale*q_i.u to every logit of row i: O unchanged,
    # LSE shifted by exactly that amount (checks the max subtraction and LSE).
    n, d, scale = 33, 8, 0.5
    q, k, v = rnd((n, d), 20), rnd((n, d), 21), rnd((n, d), 22)
    u = rnd((d,), 23) * 3.0
    for causal in (False, True):
        o1, l1 = oracle.attention_fwd(q, k, v, scale, causal)
        o2, l2 = oracle.attention_fwd(q, k + u, v, scale, causal)
        np.testing.assert_allclose(o1, o2, atol=1e-12)
        np.testing.assert_allclose(l2 - l1, scale * (q @ u), atol=1e-12)


def test_scale_folds_into_query():
    n, d = 24, 8
    q, k, v = rnd((n, d), 24), rnd((n, d), 25), rnd((n, d), 26)
    o1, l1 = oracle.attention_fwd(q, k, v, 0.125, causal=True)
    o2, l2 = oracle.attention_fwd(q * 0.125, k, v, 1.0, causal=True)
    np.testing.assert_allclose(o1, o2, atol=1e-14)
    np.testing.assert_allclose(l1, l2, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_row_weights_sum_to_one(causal):
    n, d = 45, 8
    q, k, v = rnd((n, d), 27), rnd((n, d), 28), rnd((n, d), 29)
    for i in (0, 1, 22, n - 1):
        p = oracle.row_weights(q, k, v, 0.5, causal, i)
        assert (p >= 0).all()
        assert abs(p.sum() - 1.0) < 1e-12
        if causal:
            assert (p[i + 1:] == 0).all() and (p[:i + 1] > 0).all()


def test_lse_against_library_logsumexp():
    scipy_special = pytest.importorskip("scipy.special")
    n, d, scale = 31, 16, 0.25
    q, k, v = rnd((n, d), 30), rnd((n, d), 31), rnd((n, d), 32)
    _, lse = oracle.attention_fwd(q, k, v, scale, causal=False)
    ref = scipy_special.logsumexp(scale * (q @ k.T), axis=1)
    np.testing.assert_allclose(lse, ref, atol=1e-12)
    o, _ = oracle.attention_fwd(q, k, v, scale, causal=False)
    np.testing.assert_allclose(o, scipy_special.softmax(scale * (q @ k.T), axis=1) @ v,
                               atol=1e-12)


# ---------------------------------------------------------------- brute force
@pytest.mark.parametrize("nq,nk,d,causal", [
    (16, 16, 8, False), (16, 16, 8, True), (9, 23, 4, True), (23, 9, 4, True),
    (64, 64, 16, True), (5, 64, 16, False), (1, 1, 3, True)])
def test_agrees_with_brute_force(nq, nk, d, causal):
    seed = nq * 1000 + nk * 10 + d + causal
    q, k, v = rnd((nq, d), seed), rnd((nk, d), seed + 1), rnd((nk, d), seed + 2)
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle.attention_fwd(q, k, v, scale, causal)
    ob, lb, pb = attention_brute(q.tolist(), k.tolist(), v.tolist(), scale, causal)
    np.testing.assert_allclose(o, np.array(ob), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(lb), rtol=0, atol=1e-12)
    for i in range(nq):
        if lb[i] != -math.inf:
            pw = oracle.row_weights(q, k, v, scale, causal, i)
            np.testing.assert_allclose(pw, pb[i], atol=1e-13)


# ---------------------------------------------------------------- plumbing
def test_batched_heads_row_subset_and_threads():
    B, H, n, d = 2, 3, 70, 16
    q, k, v = rnd((B, H, n, d), 40), rnd((B, H, n, d), 41), rnd((B, H, n, d), 42)
    o1, l1 = oracle.attention_fwd(q, k, v, 0.25, True, nthreads=1)
    o8, l8 = oracle.attention_fwd(q, k, v, 0.25, True, nthreads=8)
    np.testing.assert_array_equal(o1, o8)
    np.testing.assert_array_equal(l1, l8)
    rows = [0, 5, 69]
    os_, ls = oracle.attention_fwd(q, k, v, 0.25, True, rows=rows)
    np.testing.assert_array_equal(os_, o1[:, :, rows])
    np.testing.assert_array_equal(ls, l1[:, :, rows])
    # each (b, h) is its own problem
    ob, lb = oracle.attention_fwd(q[1, 2], k[1, 2], v[1, 2], 0.25, True)
    np.testing.assert_array_equal(ob, o1[1, 2])


def test_rejects_bad_rows():
    q = np.zeros((4, 2))
    with pytest.raises(ValueError):
        oracle.attention_fwd(q, q, q, 1.0, False, rows=[4])


# ---------------------------------------------------------------- workloads
def test_kv_bytes_match_pages_memory_table():
    # The pages' memory table lists the KV-cache size for batch 8, 32
    # heads, head dim 64 in fp16; the benchmark's byte accounting must
    # reproduce it (K and V, 2 bytes per element).
    rows = []
    with open(os.path.join(HERE, "golden", "kv_cache_memory.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                n, mib = line.split()
                rows.append((int(n), int(mib)))
    assert len(rows) == 4
    for n, mib in rows:
        w = W.N8192.with_(N=n, dtype="fp16")
        assert w.kv_bytes() == mib * 2 ** 20


def test_inputs_are_seeded_and_rounded():
    w = W.TINY
    q1, k1, v1 = W.make_inputs(w)
    q2, k2, v2 = W.make_inputs(w)
    assert q1.dtype == torch.float16 and q1.shape == (1, 2, 128, 64)
    assert torch.equal(q1, q2) and torch.equal(k1, k2) and torch.equal(v1, v2)
    assert not torch.equal(q1, k1)
    q8, _, _ = W.make_inputs(W.N512_Q8.with_(B=1, H=1))
    assert q8.float().abs().max() > 16.0
    assert W.N8192.flops() == 4.0 * 8 * 32 * 8192 ** 2 * 64
    assert W.N8192_CAUSAL.flops() == W.N8192.flops() / 2
    rows = W.sample_rows(32768, 256)
    assert len(rows) == 256 and rows[0] == 0 and rows[-1] == 32767
    heads = W.sample_heads(W.N8192, 4)
    assert len(set(heads)) == 4
