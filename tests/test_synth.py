"""The seeded input generators (CPU) follow the recipe their docstrings and
the design notes state: the distributions, the per-row Zipf-like bias of the
top-K workload, the synthetic cache's distinct ids, determinism by seed, and
slices of the top-K workload that match the full draw."""


import numpy as np
import pytest
import torch

from top_kl_loss_tcgen05_b300 import synth


def test_student_moments_and_logit_variance():
    T, d, V = 512, 256, 2048
    H, W = synth.student(T, d, V, seed=3)
    assert H.dtype == torch.bfloat16 and W.dtype == torch.bfloat16
    assert abs(H.float().var().item() - 1.0) < 0.02
    assert abs(W.float().var().item() * d - 1.0) < 0.02  # N(0, 1/d): variance, not std
    z = H.float() @ W.float().T
    assert abs(z.var().item() - 1.0) < 0.05  # unit-variance logits


def test_teacher_head_variance_matches_the_perturbed_teacher():
    T, d, V = 256, 256, 2048
    H, W = synth.teacher_head(T, d, V, seed=4)
    x = H.float() @ W.float().T
    assert abs(x.var().item() - 3.375) < 0.15
    Hs, Ws = synth.student(T, d, V, seed=4)
    tl = synth.teacher_logits(Hs, Ws, seed=4)
    assert abs(tl.var().item() - 1.5 ** 2 * 1.5) < 0.15  # 1.5 H (W + E)^T, E ~ N(0, 0.5/d)


def test_topk_logits_bias_and_noise():
    T, V = 300, 5000
    x = synth.topk_logits(T, V, seed=5).double()
    assert x.shape == (T, V)
    for t in (0, 17, 299):
        row = x[t]
        # the bias is 0 at one position v* and -log(1 + k) at (v* + k) mod V; find v* as the
        # offset that best explains the row, then check the residual is N(0, 2) noise
        v = torch.arange(V, dtype=torch.float64)
        best = None
        for vstar in range(V):
            b = -torch.log1p(torch.remainder(v - vstar, V))
            if best is None or (row - b).var() < best[0]:
                best = ((row - b).var().item(), vstar)
            if vstar > 0 and vstar % 1000 == 0 and best[0] < 2.3:
                break
        assert abs(best[0] - 2.0) < 0.25, best


def test_topk_logits_block_slices_match_the_full_draw():
    full = synth.topk_logits(600, 333, seed=6)
    assert torch.equal(full[256:512], synth.topk_logits(600, 333, seed=6, row0=256, rows=256))
    assert torch.equal(full[512:], synth.topk_logits(600, 333, seed=6, row0=512))  # to the end
    assert torch.equal(full[:512], synth.topk_logits(600, 333, seed=6, rows=512))
    with pytest.raises(ValueError):
        synth.topk_logits(600, 333, seed=6, row0=100)


@pytest.mark.parametrize("V,K", [(7, 7), (64, 63), (1000, 100), (4097, 16)])
def test_synthetic_cache_ids_distinct_and_logp_descending(V, K):
    ids, logp = synth.synthetic_cache(50, V, K, seed=7)
    assert ids.dtype == torch.int32 and logp.dtype == torch.float32
    assert int(ids.min()) >= 0 and int(ids.max()) < V
    s = torch.sort(ids, dim=1).values
    assert bool((s[:, 1:] != s[:, :-1]).all())
    assert bool((logp[:, 1:] <= logp[:, :-1]).all())
    with pytest.raises(ValueError):
        synth.synthetic_cache(5, V, V + 1, seed=7)


def test_generators_are_deterministic_by_seed():
    a = synth.student(64, 32, 100, seed=9)
    b = synth.student(64, 32, 100, seed=9)
    c = synth.student(64, 32, 100, seed=10)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert not torch.equal(a[0], c[0])
    i1, l1 = synth.synthetic_cache(20, 500, 10, seed=11)
    i2, l2 = synth.synthetic_cache(20, 500, 10, seed=11)
    assert torch.equal(i1, i2) and torch.equal(l1, l2)
