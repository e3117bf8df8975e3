"""Seeded random shapes through the fused loss (forward, backward and the
single call) against the fp64 oracle, cycling through the GEMM tile
configurations: one CTA per tile, CTA pairs at the default widths, all
narrow, all wide. The shapes are ragged in every dimension (T, d, V, K,
chunk), with small and tile-edge values."""

import numpy as np
import pytest
import torch

import top_kl_loss_tcgen05_b300 as kd
from oracle import kd_oracle as O
from top_kl_loss_tcgen05_b300 import synth

pytestmark = pytest.mark.gpu

MODES = [("0", None), ("1", None), ("1", "0"), ("1", "1")]


def _shapes(n=24, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        T = int(rng.choice([1, 2, int(rng.integers(3, 700))]))
        d = int(8 * rng.integers(1, 48))
        V = int(rng.choice([int(rng.integers(1, 300)), int(rng.integers(300, 5000)), 256, 512, 513]))
        K = int(min(V, rng.integers(1, 150)))
        chunk = int(rng.choice([1, int(rng.integers(2, 300)), 1024]))
        out.append((T, d, V, K, chunk, MODES[i % len(MODES)], 5000 + i))
    return out


def frob(a, b):
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(np.asarray(a, np.float64) - b) / nb) if nb > 0 else float(np.linalg.norm(a))


@pytest.mark.parametrize("T,d,V,K,chunk,mode,seed", _shapes())
def test_random_shape_matches_oracle(cuda_dev, gemm_switch, T, d, V, K, chunk, mode, seed):
    gemm_switch(mode[0], mode[1])
    H, W = synth.student(T, d, V, seed)
    ids, logp = synth.synthetic_cache(T, V, K, seed + 1)
    H, W, ids, logp = H.to(cuda_dev), W.to(cuda_dev), ids.to(cuda_dev), logp.to(cuda_dev)
    Hn, Wn = H.float().cpu().numpy(), W.float().cpu().numpy()
    i, lp = ids.cpu().numpy(), logp.cpu().numpy()
    lo, lse_o, L_o = O.fused_kl_forward(Hn, Wn, i, lp)
    dH_o, dW_o = O.fused_kl_backward(Hn, Wn, i, lp, 1.0 / T)
    loss, lse, rows = kd.fused_kl_fwd(H, W, ids, logp, chunk, want_rows=True)
    dH, dW = kd.fused_kl_bwd(H, W, ids, logp, lse, chunk, 1.0 / T)
    l1, lse1, r1, dH1, dW1 = kd.fused_kl_fwdbwd(H, W, ids, logp, chunk, want_rows=True)
    torch.cuda.synchronize()
    for lv, lsev, rv, dHv, dWv in ((loss, lse, rows, dH, dW), (l1, lse1, r1, dH1, dW1)):
        assert abs(lv.item() - lo) <= 1e-3 * abs(lo) + 1e-6
        np.testing.assert_allclose(lsev.cpu().numpy(), lse_o, rtol=1e-5, atol=1e-5)
        np.testing.assert_allclose(rv.cpu().numpy(), L_o, rtol=1e-3, atol=2e-4)
        assert frob(dHv.cpu().numpy(), dH_o) <= 1e-2
        assert frob(dWv.cpu().numpy(), dW_o) <= 1e-2


def _variant_cases(n=12, seed=4048):
    """Random shapes with a random choice of the loss variants: temperature,
    a position mask (with the mean over T or over the included positions)
    and bf16 dH."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        T = int(rng.integers(1, 900))
        d = int(8 * rng.integers(1, 40))
        V = int(rng.choice([int(rng.integers(2, 600)), int(rng.integers(600, 5000))]))
        K = int(min(V, rng.integers(1, 120)))
        chunk = int(rng.choice([1, int(rng.integers(2, 400)), 1024]))
        tau = float(rng.choice([1.0, 0.6, 2.5]))
        masked = i % 3 != 0
        over = masked and i % 2 == 0
        bf = bool(rng.integers(2))
        out.append((T, d, V, K, chunk, MODES[i % len(MODES)], 7000 + i, tau, masked, over, bf))
    return out


@pytest.mark.parametrize("T,d,V,K,chunk,mode,seed,tau,masked,over,bf", _variant_cases())
def test_random_shape_with_variants_matches_oracle(cuda_dev, gemm_switch, T, d, V, K, chunk, mode, seed, tau,
                                                   masked, over, bf):
    gemm_switch(mode[0], mode[1])
    H, W = synth.student(T, d, V, seed)
    ids, logp = synth.synthetic_cache(T, V, K, seed + 1)
    mask = None
    if masked:
        g = torch.Generator().manual_seed(seed + 2)
        mask = (torch.rand(T, generator=g) < 0.6).to(torch.uint8)
        mask[0] = 1
    Hn, Wn = H.float().numpy(), W.float().numpy()
    i, lp = ids.numpy(), logp.numpy()
    mn = None if mask is None else mask.numpy()
    lo, lse_o, L_o = O.fused_kl_forward(Hn, Wn, i, lp, temperature=tau, mask=mn, mean_over_mask=over)
    n = int((mn != 0).sum()) if (mn is not None and over) else T
    dH_o, dW_o = O.fused_kl_backward(Hn, Wn, i, lp, 1.0 / n, temperature=tau, mask=mn)
    H, W, ids, logp = H.to(cuda_dev), W.to(cuda_dev), ids.to(cuda_dev), logp.to(cuda_dev)
    md = None if mask is None else mask.to(cuda_dev)
    opts = dict(temperature=tau, mask=md, mean_over_mask=over)
    loss, lse, rows = kd.fused_kl_fwd(H, W, ids, logp, chunk, want_rows=True, **opts)
    dH, dW = kd.fused_kl_bwd(H, W, ids, logp, lse, chunk, 1.0 if over else 1.0 / T, dH_bf16=bf, **opts)
    l1, lse1, r1, dH1, dW1 = kd.fused_kl_fwdbwd(H, W, ids, logp, chunk, want_rows=True, dH_bf16=bf, **opts)
    torch.cuda.synchronize()
    for lv, lsev, rv, dHv, dWv in ((loss, lse, rows, dH, dW), (l1, lse1, r1, dH1, dW1)):
        assert dHv.dtype == (torch.bfloat16 if bf else torch.float32)
        assert abs(lv.item() - lo) <= 1e-3 * abs(lo) + 1e-6
        np.testing.assert_allclose(lsev.cpu().numpy(), lse_o, rtol=1e-5, atol=1e-5)
        np.testing.assert_allclose(rv.cpu().numpy(), L_o, rtol=1e-3, atol=2e-4)
        dHn = dHv.float().cpu().numpy()
        if mn is not None:
            assert np.all(dHn[mn == 0] == 0.0)
        assert frob(dHn, dH_o) <= 1e-2
        assert frob(dWv.cpu().numpy(), dW_o) <= 1e-2
