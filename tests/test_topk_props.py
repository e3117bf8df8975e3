"""The full-size top-K check (tests/topk_props.py) must accept the oracle's
answer and reject answers with a planted mistake."""

import numpy as np
import pytest
import torch

from oracle import kd_oracle as O
from topk_props import check_topk_rows


def _case(seed, T=9, V=300, K=20):
    rng = np.random.default_rng(seed)
    x = rng.integers(-4, 5, size=(T, V)).astype(np.float32)  # heavy ties
    x[x == 0] = np.where(rng.random(int((x == 0).sum())) < 0.5, -0.0, 0.0)
    ids, logp = O.topk_cache(x, K)
    return torch.from_numpy(x), torch.from_numpy(ids), torch.from_numpy(logp)


@pytest.mark.parametrize("seed", range(4))
def test_accepts_the_oracle(seed):
    x, ids, logp = _case(seed)
    check_topk_rows(x, ids, logp, 1e-6, block=4)


def _mutants(x, ids, logp):
    K = ids.shape[1]
    vals = torch.gather(x, 1, ids.long())
    # swap the order of two equal values
    t, j = map(int, torch.nonzero(vals[:, 1:] == vals[:, :-1])[0])
    a = ids.clone(); a[t, j], a[t, j + 1] = ids[t, j + 1], ids[t, j]
    yield "tie order", a, logp
    # drop the K-th element for the best element not chosen
    b = ids.clone()
    row = x[0].clone(); row[ids[0].long()] = -1e30
    b[0, K - 1] = int(torch.argmax(row))
    yield "K-th element replaced", b, logp
    # a tie at the K-th value goes to a higher id than the lowest
    for t in range(x.shape[0]):
        vK = x[t, ids[t, K - 1]]
        eq = torch.nonzero(x[t] == vK).flatten()
        chosen = set(ids[t].tolist())
        higher = [int(i) for i in eq if int(i) not in chosen]
        if higher:
            c = ids.clone(); c[t, K - 1] = higher[-1]
            yield "tie to a higher id", c, logp
            break
    yield "logp shifted", ids, logp + 1e-3


@pytest.mark.parametrize("seed", range(4))
def test_rejects_planted_mistakes(seed):
    x, ids, logp = _case(seed)
    n = 0
    for name, i2, l2 in _mutants(x, ids, logp):
        with pytest.raises(AssertionError):
            check_topk_rows(x, i2, l2, 1e-6, block=4)
        n += 1
    assert n >= 3
