"""kd_teacher_topk_cache (teacher hidden states + LM head -> top-K cache,
logits only ever one chunk at a time) against the fp64 oracle.

* Small-integer bf16 inputs make every fp32 logit an exact integer, so the
  ids must match the oracle bit for bit, including the heavy ties at the
  K-th place (lowest ids win).
* Gaussian inputs: the GPU logits carry fp32 rounding (about 1e-6), so
  where two oracle logits lie closer than that the order may differ. There
  the result is checked for validity: every chosen id is within EPS of the
  oracle's K-th value and in EPS-descending order. logp is compared to 1e-4.
* The fast path (tiles at or above the K-th largest tile maximum) and the
  exact radix path give identical results, and the fused path equals
  kd_topk_cache on the same fp32 logits taken from the same GEMM.
"""

import os

import numpy as np
import pytest
import torch

import top_kl_loss_tcgen05_b300 as kd
from oracle import kd_oracle as O
from top_kl_loss_tcgen05_b300 import _native, workspace

pytestmark = pytest.mark.gpu

EPS = 1e-4


def _ints(shape, seed, lo=-2, hi=2):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, shape, generator=g).to(torch.bfloat16)


def _gauss(T, d, V, seed):
    g = torch.Generator().manual_seed(seed)
    H = torch.randn(T, d, generator=g).to(torch.bfloat16)
    W = (torch.randn(V, d, generator=g) / d ** 0.5).to(torch.bfloat16)
    return H, W


def _run(H, W, K, chunk, dev):
    ids, logp = kd.teacher_topk_cache(H.to(dev), W.to(dev), K, chunk=chunk)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), logp.cpu().numpy()


@pytest.mark.parametrize("T,d,V,K,chunk", [
    (300, 64, 4096, 100, 128),   # ragged T over chunks; heavy ties at the K-th place
    (77, 32, 1000, 33, 64),      # V not a multiple of the 256-column tile
    (64, 64, 300, 100, 64),      # fewer tiles than K: every tile is read
    (50, 16, 64, 64, 32),        # K = V
])
def test_integer_logits_are_bit_exact(cuda_dev, T, d, V, K, chunk):
    H, W = _ints((T, d), T + d), _ints((V, d), V + K)
    ids, logp = _run(H, W, K, chunk, cuda_dev)
    ids_o, logp_o = O.teacher_topk_cache(H.float().numpy(), W.float().numpy(), K)
    assert np.array_equal(ids, ids_o)
    np.testing.assert_allclose(logp, logp_o, rtol=0, atol=EPS)


def test_all_equal_logits_take_the_lowest_ids(cuda_dev):
    T, d, V, K = 40, 16, 5000, 10
    H = _ints((T, d), 1)
    W = torch.zeros(V, d, dtype=torch.bfloat16)
    ids, logp = _run(H, W, K, 32, cuda_dev)
    assert np.array_equal(ids, np.tile(np.arange(K, dtype=np.int32), (T, 1)))
    np.testing.assert_allclose(logp, -np.log(V), rtol=0, atol=EPS)


def test_gaussian_logits_valid_against_oracle(cuda_dev):
    T, d, V, K = 256, 512, 50000, 100
    H, W = _gauss(T, d, V, 21)
    ids, logp = _run(H, W, K, 96, cuda_dev)
    x = H.double().numpy() @ W.double().numpy().T
    ids_o, logp_o = O.teacher_topk_cache(H.float().numpy(), W.float().numpy(), K)
    lse = np.log(np.exp(x - x.max(1, keepdims=True)).sum(1)) + x.max(1)
    exact_rows = 0
    for t in range(T):
        g = ids[t]
        assert len(set(g.tolist())) == K
        xv = x[t, g]
        assert np.all(xv[:-1] >= xv[1:] - EPS)                      # descending (up to rounding)
        kth = x[t, ids_o[t, -1]]
        assert xv.min() >= kth - EPS                                # nothing below the K-th value
        np.testing.assert_allclose(logp[t], xv - lse[t], rtol=0, atol=EPS)
        exact_rows += np.array_equal(g, ids_o[t])
    assert exact_rows >= 0.8 * T  # order differs only where oracle logits nearly tie


def test_fast_and_exact_paths_agree_and_match_topk_of_the_same_logits(cuda_dev, topk_exact):
    T, d, V, K = 200, 256, 20000, 64
    H, W = _gauss(T, d, V, 5)
    Hd, Wd = H.to(cuda_dev), W.to(cuda_dev)
    ids_f, logp_f = kd.teacher_topk_cache(Hd, Wd, K, chunk=128)
    topk_exact(True)
    ids_e, logp_e = kd.teacher_topk_cache(Hd, Wd, K, chunk=128)
    topk_exact(False)
    torch.cuda.synchronize()
    assert torch.equal(ids_f, ids_e) and torch.equal(logp_f, logp_e)
    # the same fp32 logits from the same GEMM (pair tiles, K-major operands),
    # then the logits-input top-K kernel
    X = torch.empty(T, V, dtype=torch.float32, device=cuda_dev)
    ws = workspace(256, cuda_dev)
    rc = _native.lib().kd_test_gemm(Hd.data_ptr(), Wd.data_ptr(), X.data_ptr(), T, V, d, 0, 0, 4, ws.data_ptr(),
                                    torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    ids_t, logp_t = kd.topk_cache(X, K)
    torch.cuda.synchronize()
    assert torch.equal(ids_f, ids_t)
    torch.testing.assert_close(logp_f, logp_t, rtol=0, atol=1e-5)


def test_rejects_bad_arguments_before_launch(cuda_dev):
    H = torch.zeros(8, 12, dtype=torch.bfloat16, device=cuda_dev)  # d % 8 != 0
    W = torch.zeros(100, 12, dtype=torch.bfloat16, device=cuda_dev)
    with pytest.raises(_native.KDError) as e:
        kd.teacher_topk_cache(H, W, 5)
    assert e.value.code == 2
