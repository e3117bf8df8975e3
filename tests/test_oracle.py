"""Pins for the fp64 oracle, checked against facts that come from outside it.

Each test checks the oracle against something it does not compute itself:
hand-derived closed forms, a brute-force Python sort, finite differences,
scipy/torch routines for a special case (dense KL when K = V; logsumexp), or
an invariant of the definition (Gibbs' inequality, KL = 0 when the
distributions match, teacher shift invariance). A plausible mistake in the
oracle fails at least one of them:

* wrong KL direction: closed-form (finite vs infinite) and dense KL checks.
* student renormalised over K: closed form log(3/2).
* missing teacher renormalisation: shift-invariance and dense KL checks.
* wrong sign or index in the gradient: finite differences on z, H and W.
* sum instead of mean over positions: closed-form mean and 'batchmean'.
* tie order in top-K: hand-written fixtures and the brute-force sort.
"""

import json
import math
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats
import torch

from oracle import kd_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- top-K cache


def _brute_topk(row, K):
    """Independent brute force: Python's sort on the key (-value, id)."""
    return sorted(range(len(row)), key=lambda j: (-float(row[j]), j))[:K]


def test_topk_golden_ties():
    with open(os.path.join(GOLDEN, "topk_ties.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        row = np.array([c["row"]], dtype=np.float64)
        ids, _ = O.topk_cache(row, c["K"])
        assert ids[0].tolist() == c["ids"], c


@pytest.mark.parametrize("seed", range(6))
def test_topk_matches_bruteforce_with_ties(seed):
    rng = np.random.default_rng(seed)
    T, V = 7, 53
    # small integer range -> many ties; include signed zeros
    x = rng.integers(-3, 4, size=(T, V)).astype(np.float64)
    x[x == 0] = np.where(rng.random(np.sum(x == 0)) < 0.5, -0.0, 0.0)
    for K in (1, 2, 5, 17, V):
        ids, _ = O.topk_cache(x, K)
        for t in range(T):
            assert ids[t].tolist() == _brute_topk(x[t], K)


def test_topk_logp_is_log_softmax():
    rng = np.random.default_rng(3)
    x = rng.normal(0, 2, size=(5, 300)).astype(np.float32)
    ids, logp = O.topk_cache(x, 10)
    lse = scipy.special.logsumexp(x.astype(np.float64), axis=1)
    ref = np.take_along_axis(x.astype(np.float64), ids.astype(np.int64), 1) - lse[:, None]
    assert logp.dtype == np.float32
    np.testing.assert_allclose(logp, ref, rtol=0, atol=4e-7)
    # probabilities of the full softmax at the chosen ids
    full = scipy.special.softmax(x.astype(np.float64), axis=1)
    np.testing.assert_allclose(np.exp(logp.astype(np.float64)),
                               np.take_along_axis(full, ids.astype(np.int64), 1), rtol=1e-6)


def test_logsumexp_rows_vs_scipy():
    rng = np.random.default_rng(11)
    x = rng.normal(0, 30, size=(9, 1000))
    np.testing.assert_allclose(O.logsumexp_rows(x), scipy.special.logsumexp(x, axis=1), rtol=1e-14)


def test_topk_rejects_bad_K():
    with pytest.raises(ValueError):
        O.topk_cache(np.zeros((2, 4)), 5)
    with pytest.raises(ValueError):
        O.topk_cache(np.zeros((2, 4)), 0)


# ---------------------------------------------------------------- loss


def test_closed_form_full_vocab_student():
    """V=3, teacher mass 1/2 on ids 0 and 1, student logits all 0.

    q = (1/3, 1/3, 1/3) over the full vocabulary, so
    KL(p||q) = 2 * 1/2 * log((1/2)/(1/3)) = log(3/2). A student renormalised
    over K would give 0. The reverse direction KL(q||p) would be infinite.
    The gradient is q - p = (-1/6, -1/6, 1/3).
    """
    z = np.zeros((1, 3))
    ids = np.array([[0, 1]])
    logp = np.log(np.array([[0.5, 0.5]]))
    L, lse = O.kl_rows_from_logits(z, ids, logp)
    assert L[0] == pytest.approx(math.log(1.5), rel=1e-14)
    assert lse[0] == pytest.approx(math.log(3.0), rel=1e-14)
    g = O.dlogits(z, ids, logp, 1.0)
    np.testing.assert_allclose(g[0], [-1 / 6, -1 / 6, 1 / 3], rtol=1e-13)


def test_closed_form_mean_over_positions():
    """Two positions: the first as above (log 3/2); the second has K=1 on id 2
    with z = (0, 0, log 2), so q_2 = 2/4 and L = -log(1/2) = log 2. The mean is
    (log 1.5 + log 2)/2 = log(3)/2."""
    z = np.array([[0.0, 0.0, 0.0], [0.0, 0.0, math.log(2.0)]])
    # row 2 has one real entry; its second entry carries zero teacher mass
    ids = np.array([[0, 1], [2, 2]])
    logp = np.array([[math.log(0.5), math.log(0.5)], [0.0, -1e300]])
    L, _ = O.kl_rows_from_logits(z, ids, logp)
    np.testing.assert_allclose(L, [math.log(1.5), math.log(2.0)], rtol=1e-13)
    # through the projection: H = I (d = 2) and W = z^T, so H W^T = z
    loss, _, _ = O.fused_kl_forward(np.eye(2), z.T.copy(), ids, logp)
    assert loss == pytest.approx(math.log(3.0) / 2, rel=1e-13)


def test_gibbs_nonnegative():
    rng = np.random.default_rng(5)
    T, V, K = 40, 97, 9
    z = rng.normal(0, 3, size=(T, V))
    ids = np.stack([rng.choice(V, K, replace=False) for _ in range(T)])
    logp = rng.normal(0, 2, size=(T, K))
    L, _ = O.kl_rows_from_logits(z, ids, logp)
    assert np.all(L >= -1e-12)
    assert np.all(L > 0)  # strictly: q has mass outside K


def test_kl_zero_when_student_matches_teacher():
    """z at the K ids = teacher log-probs + C, and -1e300 elsewhere (exp -> 0):
    q equals the renormalised teacher, so the KL is 0."""
    rng = np.random.default_rng(6)
    T, V, K = 8, 31, 5
    ids = np.stack([rng.choice(V, K, replace=False) for _ in range(T)])
    logp = rng.normal(-3, 1.5, size=(T, K))
    z = np.full((T, V), -1e300)
    C = rng.normal(0, 10, size=(T, 1))
    np.put_along_axis(z, ids, logp + C, axis=1)
    L, _ = O.kl_rows_from_logits(z, ids, logp)
    np.testing.assert_allclose(L, 0.0, atol=1e-13)
    g = O.dlogits(z, ids, logp, 1.0)
    np.testing.assert_allclose(g, 0.0, atol=1e-13)


def test_teacher_shift_invariance_and_normalisation():
    rng = np.random.default_rng(7)
    T, V, K = 6, 50, 7
    z = rng.normal(0, 2, size=(T, V))
    ids = np.stack([rng.choice(V, K, replace=False) for _ in range(T)])
    logp = rng.normal(0, 1, size=(T, K))
    L1, _ = O.kl_rows_from_logits(z, ids, logp)
    L2, _ = O.kl_rows_from_logits(z, ids, logp + rng.normal(0, 50, size=(T, 1)))
    np.testing.assert_allclose(L1, L2, rtol=1e-11)
    p, lp = O.teacher_probs(logp)
    np.testing.assert_allclose(p.sum(1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(np.exp(lp), p, rtol=1e-14)


def test_dense_kl_when_K_equals_V():
    """With K = V the top-K teacher is the full teacher softmax, and the loss
    must equal the textbook dense KL: torch kl_div(log q, p, 'batchmean') and
    scipy.stats.entropy(p, q) per row (the Dense KL variant)."""
    rng = np.random.default_rng(8)
    T, d, V = 12, 6, 40
    H = rng.normal(0, 1, size=(T, d))
    W = rng.normal(0, 1 / math.sqrt(d), size=(V, d))
    tlog = rng.normal(0, 2, size=(T, V))
    ids, logp = O.topk_cache(tlog, V)
    loss, lse, L = O.fused_kl_forward(H, W, ids, logp)
    z = torch.from_numpy(H @ W.T)
    logq = torch.log_softmax(z, dim=1)
    p = torch.softmax(torch.from_numpy(tlog), dim=1)
    ref = torch.nn.functional.kl_div(logq, p, reduction="batchmean").item()
    # logp is rounded to fp32 in the cache: allow that rounding
    assert loss == pytest.approx(ref, rel=1e-6)
    for t in range(T):
        assert L[t] == pytest.approx(scipy.stats.entropy(p[t].numpy(), torch.softmax(z[t], 0).numpy()), rel=1e-5)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(H @ W.T, axis=1), rtol=1e-14)


def _fd(f, x, h=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = x[i]
        x[i] = old + h
        fp = f()
        x[i] = old - h
        fm = f()
        x[i] = old
        g[i] = (fp - fm) / (2 * h)
    return g


def test_logit_gradient_matches_finite_differences():
    rng = np.random.default_rng(9)
    T, V, K = 3, 11, 4
    z = rng.normal(0, 1.5, size=(T, V))
    ids = np.stack([rng.choice(V, K, replace=False) for _ in range(T)])
    logp = rng.normal(0, 1, size=(T, K))
    fd = _fd(lambda: O.kl_rows_from_logits(z, ids, logp)[0].sum(), z)
    an = O.dlogits(z, ids, logp, 1.0)
    np.testing.assert_allclose(an, fd, rtol=1e-6, atol=1e-9)


def test_duplicate_ids_gradient_is_scatter_add():
    rng = np.random.default_rng(10)
    T, V, K = 2, 7, 4
    z = rng.normal(0, 1, size=(T, V))
    ids = np.array([[1, 1, 4, 6], [0, 3, 3, 3]])
    logp = rng.normal(0, 1, size=(T, K))
    fd = _fd(lambda: O.kl_rows_from_logits(z, ids, logp)[0].sum(), z)
    np.testing.assert_allclose(O.dlogits(z, ids, logp, 1.0), fd, rtol=1e-6, atol=1e-9)


def test_dH_dW_match_finite_differences():
    """Mean loss over T positions; scale 1/T. Finite differences on every
    entry of H and W pin dH = g W and dW = g^T H, including the transposes."""
    rng = np.random.default_rng(12)
    T, d, V, K = 4, 5, 9, 3
    H = rng.normal(0, 1, size=(T, d))
    W = rng.normal(0, 0.5, size=(V, d))
    ids = np.stack([rng.choice(V, K, replace=False) for _ in range(T)])
    logp = rng.normal(0, 1, size=(T, K))

    def loss():
        return O.fused_kl_forward(H, W, ids, logp)[0]

    fdH = _fd(loss, H)
    fdW = _fd(loss, W)
    dH, dW = O.fused_kl_backward(H, W, ids, logp, 1.0 / T)
    np.testing.assert_allclose(dH, fdH, rtol=1e-6, atol=1e-10)
    np.testing.assert_allclose(dW, fdW, rtol=1e-6, atol=1e-10)
    dH2, dW2 = O.fused_kl_backward(H, W, ids, logp, 1.0 / T, rows_per_block=3)
    np.testing.assert_allclose(dH2, dH, rtol=1e-13)
    np.testing.assert_allclose(dW2, dW, rtol=1e-13, atol=1e-16)


def test_gradient_rows_sum_to_zero():
    rng = np.random.default_rng(13)
    z = rng.normal(0, 3, size=(10, 64))
    ids = np.stack([rng.choice(64, 6, replace=False) for _ in range(10)])
    g = O.dlogits(z, ids, rng.normal(size=(10, 6)), 0.37)
    np.testing.assert_allclose(g.sum(1), 0.0, atol=1e-14)


def test_teacher_topk_cache_is_the_top_k_of_H_times_W_transposed():
    """One-hot hidden states pick single columns of the logits x = H W^T:
    row t of H = e_j gives x[t, v] = W[v, j], so the cache of row t is the
    top-K of column j of W. A transposed product or swapped operands would
    give a different, shape-incompatible or wrong answer."""
    rng = np.random.default_rng(3)
    V, d, K = 40, 6, 5
    W = rng.integers(-3, 4, size=(V, d)).astype(np.float64)  # many ties
    H = np.zeros((d, d))
    H[np.arange(d), np.arange(d)[::-1]] = 1.0  # row t selects column d-1-t
    ids, logp = O.teacher_topk_cache(H, W, K)
    for t in range(d):
        col = W[:, d - 1 - t]
        want = sorted(range(V), key=lambda v: (-col[v], v))[:K]  # value desc, id asc
        assert list(ids[t]) == want
        lse = np.log(np.exp(col).sum())
        np.testing.assert_allclose(logp[t], col[want] - lse, rtol=0, atol=1e-6)
