"""Parity at the workloads' full sizes, in the launch configuration bench.py
times (same T, d, V, K and chunk).

The full fp64 oracle over all T positions is out of reach here (up to 1e15
flops), so:
  * lse, the per-position loss L_t and dH_t are compared on a seeded sample
    of positions, for the separate calls and for the single call. It
    includes the first and last positions and chunk and group boundaries,
    and the oracle computes each sampled row on its own;
  * the scalar loss must equal the mean of the per-position losses, a
    property that holds at any size;
  * dW (a sum over all positions) is compared in full on a T-truncated run
    with the same d, V and chunk: one full backward group (G chunks, with
    G = clamp(4096 / chunk, 1, 4) as include/kd.h states) plus a ragged
    second group of 37 positions, so that the second group's dW is added to
    the first one's.
The teacher cache is synthetic (K distinct ids per row), so that no oracle
input comes from the CUDA path.
"""

import numpy as np
import pytest
import torch

import top_kl_loss_tcgen05_b300 as kd
from oracle import kd_oracle as O
from top_kl_loss_tcgen05_b300 import synth

pytestmark = pytest.mark.gpu

LOSS_RTOL = 1e-3
GRAD_RTOL = 1e-2
# Regression bound on the achieved dH / dW error (relative Frobenius). The
# contract tolerance is GRAD_RTOL = 1e-2. What the kernels achieve is set by
# one bf16 rounding of dz (relative rounding error ~2^-8 at most, about
# 1.6e-3 RMS), which dH = dz W and dW = dz^T H inherit: 1.46e-3 to 1.72e-3
# measured on B300 over the tiny, ragged and full-size cases, for the
# recompute path and the single call alike (the norm is dominated by the
# teacher-id entries, formed in fp32 and rounded once on both paths).
# GRAD_ACHIEVED is about 1.5x the largest of those: an extra rounding or a
# lost bit of the dz path fails it while the 1e-2 contract still holds.
GRAD_ACHIEVED = 2.5e-3


def frob(a, b):
    return float(np.linalg.norm(np.asarray(a, np.float64) - b) / np.linalg.norm(b))


def _inputs(name, T=None):
    c = synth.CONFIGS[name]
    T = c["T"] if T is None else T
    dev = torch.device("cuda:0")
    H, W = synth.student(T, c["d"], c["V"], c["seed"], device=dev)
    ids, logp = synth.synthetic_cache(T, c["V"], c["K"], c["seed"])
    return c, H, W, ids.to(dev), logp.to(dev)


def _sample_rows(T, chunk, n=64, seed=0):
    rng = np.random.default_rng(seed)
    G = min(4, max(1, 4096 // chunk))  # chunks per backward group (include/kd.h)
    fixed = [0, T - 1, chunk - 1, chunk, min(T - 1, 2 * chunk - 1), G * chunk - 1, G * chunk]
    rows = set(int(r) for r in fixed if 0 <= r < T)
    while len(rows) < n:
        rows.add(int(rng.integers(T)))
    return np.array(sorted(rows))


@pytest.mark.parametrize("name", ["llama3b", "gptoss20b", "long"])
def test_full_size_sampled_positions(cuda_dev, name):
    c, H, W, ids, logp = _inputs(name)
    T, chunk = c["T"], c["chunk"]
    loss, lse, rows = kd.fused_kl_fwd(H, W, ids, logp, chunk, want_rows=True)
    dH, _ = kd.fused_kl_bwd(H, W, ids, logp, lse, chunk, 1.0 / T)
    torch.cuda.synchronize()
    lse_g = lse.cpu().numpy()
    rows_g = rows.cpu().numpy().astype(np.float64)
    # scalar loss = mean of per-position losses (any size)
    assert abs(loss.item() - rows_g.mean()) <= 1e-6 * abs(rows_g.mean())
    assert np.all(np.isfinite(rows_g)) and np.all(rows_g > -1e-3)  # Gibbs: KL >= 0
    # oracle on sampled positions
    S = _sample_rows(T, chunk)
    St = torch.as_tensor(S, device=cuda_dev)
    Hs = H[St].float().cpu().numpy()
    W64 = W.float().cpu().numpy().astype(np.float64)
    ids_s, logp_s = ids[St].cpu().numpy(), logp[St].cpu().numpy()
    _, lse_o, L_o = O.fused_kl_forward(Hs, W64, ids_s, logp_s)
    dH_o, _ = O.fused_kl_backward(Hs, W64, ids_s, logp_s, 1.0 / T)
    np.testing.assert_allclose(lse_g[S], lse_o, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(rows_g[S], L_o, rtol=LOSS_RTOL, atol=1e-4)
    assert abs(rows_g[S].mean() - L_o.mean()) <= LOSS_RTOL * abs(L_o.mean())
    assert frob(dH[St].cpu().numpy(), dH_o) <= GRAD_RTOL
    assert frob(dH[St].cpu().numpy(), dH_o) <= GRAD_ACHIEVED
    # the single call (no recompute) on the same positions
    del dH
    l1, lse1, rows1, dH1, dW1 = kd.fused_kl_fwdbwd(H, W, ids, logp, chunk, want_rows=True)
    torch.cuda.synchronize()
    r1 = rows1.cpu().numpy().astype(np.float64)
    assert abs(l1.item() - r1.mean()) <= 1e-6 * abs(r1.mean())
    np.testing.assert_allclose(lse1.cpu().numpy()[S], lse_o, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(r1[S], L_o, rtol=LOSS_RTOL, atol=1e-4)
    assert frob(dH1[St].cpu().numpy(), dH_o) <= GRAD_RTOL
    assert frob(dH1[St].cpu().numpy(), dH_o) <= GRAD_ACHIEVED


@pytest.mark.parametrize("name", ["llama3b", "gptoss20b", "long"])
def test_full_width_dW_on_truncated_run(cuda_dev, name):
    c = synth.CONFIGS[name]
    chunk = c["chunk"]
    G = min(4, max(1, 4096 // chunk))  # chunks per backward group (include/kd.h)
    Tp = G * chunk + 37
    c, H, W, ids, logp = _inputs(name, T=Tp)
    _, lse, _ = kd.fused_kl_fwd(H, W, ids, logp, chunk)
    dH, dW = kd.fused_kl_bwd(H, W, ids, logp, lse, chunk, 1.0 / Tp)
    torch.cuda.synchronize()
    # oracle: dW = sum_t g_t h_t^T, positions in blocks of 256 (host memory)
    H64 = H.float().cpu().numpy().astype(np.float64)
    W64 = W.float().cpu().numpy().astype(np.float64)
    idn, lpn = ids.cpu().numpy(), logp.cpu().numpy()
    dW_o = np.zeros_like(W64)
    dH_o = np.empty_like(H64)
    for t0 in range(0, Tp, 256):
        t1 = min(Tp, t0 + 256)
        z = O.student_logits(H64[t0:t1], W64)
        g = O.dlogits(z, idn[t0:t1], lpn[t0:t1], 1.0 / Tp)
        dW_o += g.T @ H64[t0:t1]
        dH_o[t0:t1] = g @ W64
    assert frob(dW.cpu().numpy(), dW_o) <= GRAD_RTOL
    assert frob(dW.cpu().numpy(), dW_o) <= GRAD_ACHIEVED
    assert frob(dH.cpu().numpy(), dH_o) <= GRAD_RTOL
    assert frob(dH.cpu().numpy(), dH_o) <= GRAD_ACHIEVED


def test_teacher_cache_full_size_sampled(cuda_dev):
    """The teacher-side cache at the bench's size (Llama-3.1-8B-shaped head,
    T=8192, d=4096, V=128256, K=100, chunk=1024): sampled positions against
    the oracle on fp64 logits. Where oracle logits lie within EPS of each
    other the fp32 order may differ, so the check is validity: every chosen
    id at or above the oracle's K-th value (up to EPS), descending up to EPS,
    and logp within 1e-4."""
    c = synth.CONFIGS["teacher"]
    T, d, V, K, chunk = c["T"], c["d"], c["V"], c["K"], c["chunk"]
    H, W = synth.teacher_head(T, d, V, c["seed"], device=cuda_dev)
    ids, logp = kd.teacher_topk_cache(H, W, K, chunk=chunk)
    torch.cuda.synchronize()
    S = _sample_rows(T, chunk, n=48, seed=7)
    Hs = H[torch.as_tensor(S, device=cuda_dev)].float().cpu().numpy().astype(np.float64)
    W64 = W.float().cpu().numpy().astype(np.float64)
    x = Hs @ W64.T
    ids_o, logp_o = O.topk_cache(x, K)
    lse = np.log(np.exp(x - x.max(1, keepdims=True)).sum(1)) + x.max(1)
    g_ids, g_lp = ids.cpu().numpy()[S], logp.cpu().numpy()[S]
    eps = 1e-4
    exact = 0
    for r in range(len(S)):
        xv = x[r, g_ids[r]]
        assert len(set(g_ids[r].tolist())) == K
        assert np.all(xv[:-1] >= xv[1:] - eps)
        assert xv.min() >= x[r, ids_o[r, -1]] - eps
        np.testing.assert_allclose(g_lp[r], xv - lse[r], rtol=0, atol=eps)
        exact += np.array_equal(g_ids[r], ids_o[r])
    assert exact >= 0.8 * len(S)


def test_group_one_at_llama3b_shape(cuda_dev):
    """group = 1 (kd_kl_options.group): every GEMM launch covers one chunk of
    1024 positions at the Llama-3.2-3B shape. Per-position results (lse, L_t,
    dH) do not depend on the grouping at all; dW differs from the default
    grouping by summation order only; both match the oracle. T-truncated to
    two chunks plus a ragged tail of 37 positions."""
    c = synth.CONFIGS["llama3b"]
    chunk = c["chunk"]
    Tp = 2 * chunk + 37
    c, H, W, ids, logp = _inputs("llama3b", T=Tp)
    ws1 = kd.fused_kl_workspace(c["d"], c["V"], c["K"], chunk, cuda_dev, group=1)
    assert ws1.numel() < kd.fused_kl_workspace(c["d"], c["V"], c["K"], chunk, cuda_dev).numel() / 3
    l1, lse1, r1 = kd.fused_kl_fwd(H, W, ids, logp, chunk, ws=ws1, want_rows=True, group=1)
    dH1, dW1 = kd.fused_kl_bwd(H, W, ids, logp, lse1, chunk, 1.0 / Tp, ws=ws1, group=1)
    l0, lse0, r0 = kd.fused_kl_fwd(H, W, ids, logp, chunk, want_rows=True)
    dH0, dW0 = kd.fused_kl_bwd(H, W, ids, logp, lse0, chunk, 1.0 / Tp)
    torch.cuda.synchronize()
    assert kd.read_device_status(ws1) == 0
    assert torch.equal(lse1, lse0) and torch.equal(r1, r0) and torch.equal(dH1, dH0)
    assert abs(l1.item() - l0.item()) <= 1e-6 * abs(l0.item())
    assert frob(dW1.cpu().numpy(), dW0.cpu().numpy().astype(np.float64)) <= 1e-5
    H64 = H.float().cpu().numpy().astype(np.float64)
    W64 = W.float().cpu().numpy().astype(np.float64)
    idn, lpn = ids.cpu().numpy(), logp.cpu().numpy()
    dW_o = np.zeros_like(W64)
    dH_o = np.empty_like(H64)
    for t0 in range(0, Tp, 256):
        t1 = min(Tp, t0 + 256)
        z = O.student_logits(H64[t0:t1], W64)
        g = O.dlogits(z, idn[t0:t1], lpn[t0:t1], 1.0 / Tp)
        dW_o += g.T @ H64[t0:t1]
        dH_o[t0:t1] = g @ W64
    assert frob(dW1.cpu().numpy(), dW_o) <= GRAD_RTOL
    assert frob(dW1.cpu().numpy(), dW_o) <= GRAD_ACHIEVED
    assert frob(dH1.cpu().numpy(), dH_o) <= GRAD_RTOL
    assert frob(dH1.cpu().numpy(), dH_o) <= GRAD_ACHIEVED
    # the single call with group = 1 on the same workspace: per position the
    # same as the single call with the default group (its epilogue takes the
    # tile maximum first, so its lse rounds differently from the forward's)
    l2, lse2, _, dH2, dW2 = kd.fused_kl_fwdbwd(H, W, ids, logp, chunk, ws=ws1, group=1)
    l3, lse3, _, dH3, dW3 = kd.fused_kl_fwdbwd(H, W, ids, logp, chunk)
    torch.cuda.synchronize()
    assert torch.equal(lse2, lse3) and torch.equal(dH2, dH3)
    assert frob(dW2.cpu().numpy(), dW3.cpu().numpy().astype(np.float64)) <= 1e-5
    np.testing.assert_allclose(lse2.cpu().numpy(), lse0.cpu().numpy(), rtol=1e-6, atol=1e-6)
    assert abs(l2.item() - l0.item()) <= 1e-5 * abs(l0.item())
    assert frob(dW2.cpu().numpy(), dW_o) <= GRAD_RTOL
    assert frob(dW2.cpu().numpy(), dW_o) <= GRAD_ACHIEVED
    assert frob(dH2.cpu().numpy(), dH_o) <= GRAD_RTOL
    assert frob(dH2.cpu().numpy(), dH_o) <= GRAD_ACHIEVED


def test_full_size_variants_sampled_positions(cuda_dev):
    """The loss variants at the GPT-OSS-20B shape (T=32768, d=2880, V=201088,
    K=100, chunk=2048): temperature 2, a seeded mask that drops about one
    position in ten, and the mean over the included positions. Sampled rows
    (masked and unmasked among them) against the oracle computing those rows
    alone: lse of z / tau, L_t (0 where masked) and dH_t (with the factor
    1/N of the full mask); the scalar loss is the sum of the rows over N."""
    c, H, W, ids, logp = _inputs("gptoss20b")
    T, chunk, tau = c["T"], c["chunk"], 2.0
    g = torch.Generator().manual_seed(77)
    mask = (torch.rand(T, generator=g) >= 0.1).to(torch.uint8)
    N = int(mask.sum())
    m_dev = mask.to(cuda_dev)
    loss, lse, rows = kd.fused_kl_fwd(H, W, ids, logp, chunk, want_rows=True, temperature=tau, mask=m_dev,
                                      mean_over_mask=True)
    dH, _ = kd.fused_kl_bwd(H, W, ids, logp, lse, chunk, 1.0, temperature=tau, mask=m_dev, mean_over_mask=True)
    torch.cuda.synchronize()
    rows_g = rows.cpu().numpy().astype(np.float64)
    assert abs(loss.item() - rows_g.sum() / N) <= 1e-6 * abs(loss.item())
    S = _sample_rows(T, chunk, n=48, seed=3)
    mk = mask.numpy()
    S = np.unique(np.concatenate([S, np.nonzero(mk == 0)[0][:8]]))  # some excluded positions too
    St = torch.as_tensor(S, device=cuda_dev)
    Hs = H[St].float().cpu().numpy()
    W64 = W.float().cpu().numpy().astype(np.float64)
    ids_s, logp_s = ids[St].cpu().numpy(), logp[St].cpu().numpy()
    _, lse_o, L_o = O.fused_kl_forward(Hs, W64, ids_s, logp_s, temperature=tau, mask=mk[S])
    dH_o, _ = O.fused_kl_backward(Hs, W64, ids_s, logp_s, 1.0 / N, temperature=tau, mask=mk[S])
    np.testing.assert_allclose(lse.cpu().numpy()[S], lse_o, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(rows_g[S], L_o, rtol=LOSS_RTOL, atol=1e-4)
    assert np.all(rows_g[S][mk[S] == 0] == 0.0)
    dH_s = dH[St].cpu().numpy()
    assert np.all(dH_s[mk[S] == 0] == 0.0)
    assert frob(dH_s, dH_o) <= GRAD_RTOL
    assert frob(dH_s, dH_o) <= GRAD_ACHIEVED
