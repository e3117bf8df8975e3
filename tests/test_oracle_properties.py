"""Property checks of the fp64 oracle on generated inputs (hypothesis).

The fixed-seed pins in test_oracle.py tie the oracle to closed forms, brute
force, library routines and finite differences. These check the same
definition over many small random cases, each against a fact that holds for
any input:

* the order of a cache row's (id, logp) entries does not matter (the C ABI
  accepts them in any order);
* adding a constant to a row of student logits changes neither the loss nor
  its gradient (the softmax is shift invariant);
* Gibbs' inequality: every per-position KL is >= 0;
* the logit gradient of every row sums to zero (q and p both sum to one);
* the gradient matches a central finite difference along a random direction;
* the tempered loss at tau is the plain loss of z / tau against the cached
  log-probs / tau (the reading of the temperature variant);
* top-K on small integer rows (heavy ties, signed zeros) equals a brute-force
  sort by (value descending, id ascending).
"""

import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

from oracle import kd_oracle as O  # noqa: E402

SETTINGS = settings(max_examples=60, deadline=None, derandomize=True)


def kl(z, ids, logp, **kw):
    """Per-position KL L_t (the first output of the oracle's logit-level loss)."""
    return O.kl_rows_from_logits(z, ids, logp, **kw)[0]


@st.composite
def problems(draw, max_T=4, max_V=24):
    """(z [T, V], ids [T, K] distinct per row, logp [T, K]) in fp64."""
    T = draw(st.integers(1, max_T))
    V = draw(st.integers(2, max_V))
    K = draw(st.integers(1, V))
    seed = draw(st.integers(0, 2**31 - 1))
    rng = np.random.default_rng(seed)
    z = rng.normal(0.0, draw(st.sampled_from([0.5, 1.0, 3.0])), size=(T, V))
    ids = np.stack([rng.permutation(V)[:K] for _ in range(T)]).astype(np.int32)
    logp = rng.normal(0.0, 2.0, size=(T, K)) - np.log(V)
    return z, ids, logp.astype(np.float32), rng


@SETTINGS
@given(problems())
def test_entry_order_within_a_row_does_not_matter(p):
    z, ids, logp, rng = p
    perm = np.stack([rng.permutation(ids.shape[1]) for _ in range(ids.shape[0])])
    ids2 = np.take_along_axis(ids, perm, axis=1)
    logp2 = np.take_along_axis(logp, perm, axis=1)
    np.testing.assert_allclose(kl(z, ids2, logp2), kl(z, ids, logp),
                               rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(O.dlogits(z, ids2, logp2, 0.5), O.dlogits(z, ids, logp, 0.5), rtol=1e-12,
                               atol=1e-14)


@SETTINGS
@given(problems(), st.floats(-50.0, 50.0))
def test_student_logit_shift_changes_nothing(p, c):
    z, ids, logp, _ = p
    shift = c * np.arange(1, z.shape[0] + 1)[:, None]  # a different constant per row
    np.testing.assert_allclose(kl(z + shift, ids, logp), kl(z, ids, logp),
                               rtol=1e-9, atol=1e-9)
    np.testing.assert_allclose(O.dlogits(z + shift, ids, logp, 1.0), O.dlogits(z, ids, logp, 1.0), rtol=1e-9,
                               atol=1e-12)


@SETTINGS
@given(problems())
def test_gibbs_and_gradient_rows_sum_to_zero(p):
    z, ids, logp, _ = p
    assert np.all(kl(z, ids, logp) >= -1e-12)
    g = O.dlogits(z, ids, logp, 1.0)
    np.testing.assert_allclose(g.sum(axis=1), 0.0, atol=1e-12)


@SETTINGS
@given(problems(max_T=3, max_V=16))
def test_gradient_matches_a_directional_finite_difference(p):
    z, ids, logp, rng = p
    T = z.shape[0]
    v = rng.normal(size=z.shape)
    h = 1e-5

    def loss(zz):
        return kl(zz, ids, logp).mean()

    fd = (loss(z + h * v) - loss(z - h * v)) / (2 * h)
    an = float(np.sum(O.dlogits(z, ids, logp, 1.0 / T) * v))
    assert abs(fd - an) <= 1e-6 * max(1.0, abs(an))


@SETTINGS
@given(problems(), st.floats(0.25, 8.0))
def test_tempered_loss_is_the_plain_loss_of_scaled_inputs(p, tau):
    z, ids, logp, _ = p
    lp64 = logp.astype(np.float64)
    np.testing.assert_allclose(kl(z, ids, lp64, temperature=tau),
                               kl(z / tau, ids, lp64 / tau), rtol=1e-10, atol=1e-12)
    # and the gradient gains exactly the chain-rule factor 1 / tau
    np.testing.assert_allclose(O.dlogits(z, ids, lp64, 1.0, temperature=tau),
                               O.dlogits(z / tau, ids, lp64 / tau, 1.0) / tau, rtol=1e-10, atol=1e-14)


@SETTINGS
@given(st.integers(1, 6), st.integers(1, 40), st.integers(0, 2**31 - 1))
def test_topk_on_integer_rows_matches_a_brute_force_sort(T, V, seed):
    rng = np.random.default_rng(seed)
    x = rng.integers(-3, 4, size=(T, V)).astype(np.float32)
    x[x == 0] = np.where(rng.random(int((x == 0).sum())) < 0.5, -0.0, 0.0)
    K = int(rng.integers(1, V + 1))
    ids, _ = O.topk_cache(x, K)
    for t in range(T):
        brute = sorted(range(V), key=lambda j: (-float(x[t, j]), j))[:K]
        assert ids[t].tolist() == brute
