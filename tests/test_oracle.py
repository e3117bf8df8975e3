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


# ------------------------------------------------------- temperature and mask


def test_temperature_limit_is_log_V_over_K():
    """As tau grows, the tempered teacher tends to uniform over its K ids and
    the tempered student to uniform over V, so L -> log(V / K). A missing
    division of z or of the teacher log-probs by tau would not converge."""
    rng = np.random.default_rng(20)
    T, V, K = 3, 50, 7
    z = rng.normal(0, 2, size=(T, V))
    ids = np.stack([rng.choice(V, K, replace=False) for _ in range(T)])
    logp = rng.normal(0, 2, size=(T, K))
    L, _ = O.kl_rows_from_logits(z, ids, logp, temperature=1e6)
    np.testing.assert_allclose(L, math.log(V / K), rtol=0, atol=1e-5)


def test_temperature_keeps_gibbs_and_kl_zero():
    """KL >= 0 at every tau, and = 0 when the tempered student equals the
    tempered teacher: z = logp on the K ids (and -inf elsewhere)."""
    rng = np.random.default_rng(21)
    T, V, K = 4, 30, 6
    ids = np.stack([rng.choice(V, K, replace=False) for _ in range(T)])
    logp = rng.normal(0, 1, size=(T, K))
    for tau in (0.3, 1.0, 2.5):
        z = rng.normal(0, 2, size=(T, V))
        L, _ = O.kl_rows_from_logits(z, ids, logp, temperature=tau)
        assert np.all(L >= -1e-12)
        z0 = np.full((T, V), -1e300)
        z0[np.arange(T)[:, None], ids] = logp + 3.0  # any shift: softmax is shift-invariant
        L0, _ = O.kl_rows_from_logits(z0, ids, logp, temperature=tau)
        np.testing.assert_allclose(L0, 0.0, atol=1e-12)


@pytest.mark.parametrize("tau", [0.7, 2.5])
def test_tempered_gradient_matches_finite_differences(tau):
    """dL/dz = (1/tau) (q_tau - p_tau): a dropped 1/tau fails."""
    rng = np.random.default_rng(22)
    T, V, K = 3, 11, 4
    z = rng.normal(0, 1.5, size=(T, V))
    ids = np.stack([rng.choice(V, K, replace=False) for _ in range(T)])
    logp = rng.normal(0, 1, size=(T, K))
    fd = _fd(lambda: O.kl_rows_from_logits(z, ids, logp, temperature=tau)[0].sum(), z)
    np.testing.assert_allclose(O.dlogits(z, ids, logp, 1.0, temperature=tau), fd, rtol=1e-6, atol=1e-9)


def test_mask_excludes_positions_and_normalises_over_the_rest():
    """The masked loss is the loss of the included positions alone (computed
    without a mask on that subset); excluded rows of dH are zero; dW is the
    subset's dW; finite differences on H and W pin the 1/N normalisation."""
    rng = np.random.default_rng(23)
    T, d, V, K = 6, 5, 9, 3
    H = rng.normal(0, 1, size=(T, d))
    W = rng.normal(0, 0.5, size=(V, d))
    ids = np.stack([rng.choice(V, K, replace=False) for _ in range(T)])
    logp = rng.normal(0, 1, size=(T, K))
    mask = np.array([1, 0, 1, 1, 0, 1], dtype=np.uint8)
    keep = mask.astype(bool)
    n = int(keep.sum())
    loss_n, lse, L = O.fused_kl_forward(H, W, ids, logp, mask=mask, mean_over_mask=True)
    loss_sub, lse_sub, L_sub = O.fused_kl_forward(H[keep], W, ids[keep], logp[keep])
    assert abs(loss_n - loss_sub) <= 1e-14 * abs(loss_sub)
    np.testing.assert_array_equal(L[~keep], 0.0)
    np.testing.assert_allclose(L[keep], L_sub, rtol=1e-14)
    loss_T, _, _ = O.fused_kl_forward(H, W, ids, logp, mask=mask, mean_over_mask=False)
    assert abs(loss_T - loss_sub * n / T) <= 1e-14 * abs(loss_T)
    dH, dW = O.fused_kl_backward(H, W, ids, logp, 1.0 / n, mask=mask)
    dH_sub, dW_sub = O.fused_kl_backward(H[keep], W, ids[keep], logp[keep], 1.0 / n)
    np.testing.assert_array_equal(dH[~keep], 0.0)
    np.testing.assert_allclose(dH[keep], dH_sub, rtol=1e-13)
    np.testing.assert_allclose(dW, dW_sub, rtol=1e-13, atol=1e-16)

    def loss():
        return O.fused_kl_forward(H, W, ids, logp, mask=mask, mean_over_mask=True)[0]

    np.testing.assert_allclose(dH, _fd(loss, H), rtol=1e-6, atol=1e-10)
    np.testing.assert_allclose(dW, _fd(loss, W), rtol=1e-6, atol=1e-10)
    lossz, _, Lz = O.fused_kl_forward(H, W, ids, logp, mask=np.zeros(T), mean_over_mask=True)
    assert lossz == 0.0 and np.all(Lz == 0.0)


def test_tempered_masked_dH_dW_match_finite_differences():
    rng = np.random.default_rng(24)
    T, d, V, K, tau = 4, 4, 8, 3, 1.7
    H = rng.normal(0, 1, size=(T, d))
    W = rng.normal(0, 0.5, size=(V, d))
    ids = np.stack([rng.choice(V, K, replace=False) for _ in range(T)])
    logp = rng.normal(0, 1, size=(T, K))
    mask = np.array([1, 1, 0, 1])

    def loss():
        return O.fused_kl_forward(H, W, ids, logp, temperature=tau, mask=mask, mean_over_mask=False)[0]

    dH, dW = O.fused_kl_backward(H, W, ids, logp, 1.0 / T, temperature=tau, mask=mask)
    np.testing.assert_allclose(dH, _fd(loss, H), rtol=1e-6, atol=1e-10)
    np.testing.assert_allclose(dW, _fd(loss, W), rtol=1e-6, atol=1e-10)
