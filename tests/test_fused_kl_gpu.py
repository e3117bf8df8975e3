"""Fused chunked KL loss (kd_fused_kl_fwd / kd_fused_kl_bwd) against the fp64
oracle on the same seeded inputs.

Tolerances: loss relative 1e-3; dH and dW relative Frobenius 1e-2 (bf16
inputs, fp32 accumulation, dz rounded to bf16 once). The per-position lse and
loss rows are checked tighter. They come from fp32 sums over V terms.
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


@pytest.fixture(params=[("0", None), ("1", None), ("1", "0"), ("1", "1")],
                ids=["cta1", "cta2", "cta2-narrow", "cta2-wide"], autouse=True)
def gemm_tiles(request, gemm_switch):
    """Every test runs with one CTA per GEMM tile, with CTA-pair tiles at the
    per-kernel default widths, and with every pair GEMM narrow or wide."""
    cta2, wide = request.param
    gemm_switch(cta2, wide)
    return request.param


def frob(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def gpu_run(H, W, ids, logp, chunk, ws=None):
    T = H.shape[0]
    loss, lse, rows = kd.fused_kl_fwd(H, W, ids, logp, chunk, ws=ws, want_rows=True)
    dH, dW = kd.fused_kl_bwd(H, W, ids, logp, lse, chunk, 1.0 / T, ws=ws)
    torch.cuda.synchronize()
    return dict(loss=loss.item(), lse=lse.cpu().numpy(), rows=rows.cpu().numpy(), dH=dH.cpu().numpy(),
                dW=dW.cpu().numpy())


def oracle_run(H, W, ids, logp):
    Hn = H.float().cpu().numpy()
    Wn = W.float().cpu().numpy()
    i = ids.cpu().numpy()
    lp = logp.cpu().numpy()
    loss, lse, L = O.fused_kl_forward(Hn, Wn, i, lp)
    dH, dW = O.fused_kl_backward(Hn, Wn, i, lp, 1.0 / Hn.shape[0])
    return dict(loss=loss, lse=lse, rows=L, dH=dH, dW=dW)


def compare(g, o):
    assert abs(g["loss"] - o["loss"]) <= LOSS_RTOL * abs(o["loss"]), (g["loss"], o["loss"])
    np.testing.assert_allclose(g["lse"], o["lse"], rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(g["rows"], o["rows"], rtol=1e-3, atol=2e-4)
    assert frob(g["dH"], o["dH"]) <= GRAD_RTOL
    assert frob(g["dH"], o["dH"]) <= GRAD_ACHIEVED
    assert frob(g["dW"], o["dW"]) <= GRAD_RTOL
    assert frob(g["dW"], o["dW"]) <= GRAD_ACHIEVED


def tiny_inputs(dev):
    c = synth.CONFIGS["tiny"]
    H, W = synth.student(c["T"], c["d"], c["V"], c["seed"])
    tl = synth.teacher_logits(H, W, c["seed"])
    ids, logp = O.topk_cache(tl.numpy(), c["K"])  # the cache comes from the oracle
    return (H.to(dev), W.to(dev), torch.from_numpy(ids).to(dev), torch.from_numpy(logp).to(dev), c["chunk"])


def test_tiny_config_matches_oracle(cuda_dev):
    H, W, ids, logp, chunk = tiny_inputs(cuda_dev)
    g = gpu_run(H, W, ids, logp, chunk)
    o = oracle_run(H, W, ids, logp)
    compare(g, o)
    assert g["loss"] > 0


def test_chunk_size_changes_only_rounding_and_runs_are_bitwise_reproducible(cuda_dev):
    H, W, ids, logp, _ = tiny_inputs(cuda_dev)
    ref = gpu_run(H, W, ids, logp, 64)
    again = gpu_run(H, W, ids, logp, 64)
    for k in ref:
        assert np.array_equal(np.asarray(ref[k]), np.asarray(again[k])), k
    for chunk in (37, 100, 128, 256, 1000):
        g = gpu_run(H, W, ids, logp, chunk)
        # per-position results do not depend on the chunk at all
        assert np.array_equal(g["lse"], ref["lse"])
        assert np.array_equal(g["rows"], ref["rows"])
        assert np.array_equal(g["dH"], ref["dH"])
        assert abs(g["loss"] - ref["loss"]) <= 1e-6 * abs(ref["loss"])
        assert frob(g["dW"], ref["dW"]) <= 1e-5


def _cache(T, V, K, seed, dev, edge=True):
    ids, logp = synth.synthetic_cache(T, V, K, seed)
    if edge:
        # ids on vocabulary-tile edges and at both ends of the vocabulary
        edges = [0, V - 1, 255 % V, 256 % V, 511 % V, 63 % V, 64 % V]
        for t in range(0, T, 3):
            row = ids[t].tolist()
            for e in edges:
                if e not in row:
                    row[np.random.default_rng(t + e).integers(K)] = e
            ids[t] = torch.tensor(row, dtype=torch.int32)
    return ids.to(dev), logp.to(dev)


@pytest.mark.parametrize("T,d,V,K,chunk", [
    (300, 264, 1000, 7, 128),     # ragged T, d (not a multiple of 64 or 192), V
    (129, 72, 4099, 33, 64),      # K-dim smaller than one 128-wide block in dW
    (64, 520, 257, 5, 64),        # V = one full logits tile + 1
    (77, 8, 31, 3, 16),           # tiny d and V
    (300, 960, 1000, 7, 128),     # d a multiple of 480, not of 512: dW in 480-wide tiles
])
def test_ragged_shapes_match_oracle(cuda_dev, T, d, V, K, chunk):
    H, W = synth.student(T, d, V, seed=T * 7 + d)
    ids, logp = _cache(T, V, K, seed=V, dev=cuda_dev)
    H, W = H.to(cuda_dev), W.to(cuda_dev)
    compare(gpu_run(H, W, ids, logp, chunk), oracle_run(H, W, ids, logp))


def test_K_equals_V_is_dense_kl(cuda_dev):
    """With K = V the teacher is the full softmax: the fused loss is the Dense
    KL variant of the same loss."""
    c = synth.CONFIGS["tiny"]
    T, d, V = 128, c["d"], c["V"]
    H, W = synth.student(T, d, V, c["seed"])
    tl = synth.teacher_logits(H, W, c["seed"])
    ids, logp = O.topk_cache(tl.numpy(), V)
    H, W = H.to(cuda_dev), W.to(cuda_dev)
    ids, logp = torch.from_numpy(ids).to(cuda_dev), torch.from_numpy(logp).to(cuda_dev)
    compare(gpu_run(H, W, ids, logp, 64), oracle_run(H, W, ids, logp))


def test_duplicate_ids_are_summed(cuda_dev):
    T, d, V, K = 96, 128, 700, 6
    H, W = synth.student(T, d, V, seed=11)
    ids, logp = synth.synthetic_cache(T, V, K, seed=12)
    ids[:, 1] = ids[:, 0]
    ids[::2, 5] = ids[::2, 0]
    H, W, ids, logp = H.to(cuda_dev), W.to(cuda_dev), ids.to(cuda_dev), logp.to(cuda_dev)
    compare(gpu_run(H, W, ids, logp, 64), oracle_run(H, W, ids, logp))


def test_bad_id_is_reported_in_status_word(cuda_dev):
    T, d, V, K = 64, 64, 512, 4
    H, W = synth.student(T, d, V, seed=1)
    ids, logp = synth.synthetic_cache(T, V, K, seed=2)
    ids[5, 2] = V  # out of range
    H, W, ids, logp = H.to(cuda_dev), W.to(cuda_dev), ids.to(cuda_dev), logp.to(cuda_dev)
    ws = kd.fused_kl_workspace(d, V, K, 32, cuda_dev)
    kd.fused_kl_fwd(H, W, ids, logp, 32, ws=ws)
    assert kd.read_device_status(ws) == 6
    assert kd.read_device_status(ws) == 0  # reading clears it
    ids[5, 2] = 0 if int(ids[5].min()) != 0 else 1
    kd.fused_kl_fwd(H, W, ids, logp, 32, ws=ws)
    assert kd.read_device_status(ws) == 0


def test_grad_scale_and_accumulate(cuda_dev):
    H, W, ids, logp, chunk = tiny_inputs(cuda_dev)
    T = H.shape[0]
    _, lse, _ = kd.fused_kl_fwd(H, W, ids, logp, chunk)
    dH1, dW1 = kd.fused_kl_bwd(H, W, ids, logp, lse, chunk, 1.0 / T)
    two = torch.tensor(2.0, device=cuda_dev)
    dH2, dW2 = kd.fused_kl_bwd(H, W, ids, logp, lse, chunk, 1.0 / T, grad_scale_dev=two)
    torch.testing.assert_close(dH2, 2 * dH1, rtol=1e-2, atol=1e-6)
    torch.testing.assert_close(dW2, 2 * dW1, rtol=1e-2, atol=1e-6)
    dW3 = dW1.clone()
    kd.fused_kl_bwd(H, W, ids, logp, lse, chunk, 1.0 / T, dW=dW3, accumulate_dW=True)
    torch.testing.assert_close(dW3, 2 * dW1, rtol=1e-5, atol=1e-7)


def test_autograd_function(cuda_dev):
    H, W, ids, logp, chunk = tiny_inputs(cuda_dev)
    o = oracle_run(H, W, ids, logp)
    Hg = H.clone().requires_grad_(True)
    Wg = W.clone().requires_grad_(True)
    loss = kd.FusedKL.apply(Hg, Wg, ids, logp, chunk)
    (3.0 * loss).backward()
    assert abs(loss.item() - o["loss"]) <= LOSS_RTOL * abs(o["loss"])
    assert frob(Hg.grad.float().cpu().numpy(), 3.0 * o["dH"]) <= GRAD_RTOL
    assert frob(Wg.grad.float().cpu().numpy(), 3.0 * o["dW"]) <= GRAD_RTOL
