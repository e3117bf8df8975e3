"""kd_fused_kl_fwdbwd (forward and backward in one call, each chunk's logits
computed once) against the fp64 oracle on the same seeded inputs, and against
the separate forward + backward calls.

Tolerances are those of the separate calls: loss relative 1e-3, dH and dW
relative Frobenius 1e-2. dz off the teacher ids is rounded to bf16 twice
here (e = exp(z - m_tile), then dz), about 2^-8 relative per element, well
inside 1e-2 in Frobenius norm.
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


def one_call(H, W, ids, logp, chunk, **kw):
    loss, lse, rows, dH, dW = kd.fused_kl_fwdbwd(H, W, ids, logp, chunk, want_rows=True, **kw)
    torch.cuda.synchronize()
    return dict(loss=loss.item(), lse=lse.cpu().numpy(), rows=rows.cpu().numpy(), dH=dH.cpu().numpy(),
                dW=dW.cpu().numpy())


def oracle_run(H, W, ids, logp):
    Hn, Wn = H.float().cpu().numpy(), W.float().cpu().numpy()
    i, lp = ids.cpu().numpy(), logp.cpu().numpy()
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
    ids, logp = O.topk_cache(tl.numpy(), c["K"])
    return (H.to(dev), W.to(dev), torch.from_numpy(ids).to(dev), torch.from_numpy(logp).to(dev), c["chunk"])


def test_tiny_config_matches_oracle(cuda_dev):
    H, W, ids, logp, chunk = tiny_inputs(cuda_dev)
    compare(one_call(H, W, ids, logp, chunk), oracle_run(H, W, ids, logp))


def test_matches_separate_calls_and_is_reproducible(cuda_dev):
    H, W, ids, logp, chunk = tiny_inputs(cuda_dev)
    T = H.shape[0]
    a = one_call(H, W, ids, logp, chunk)
    b = one_call(H, W, ids, logp, chunk)
    for k in a:
        assert np.array_equal(np.asarray(a[k]), np.asarray(b[k])), k
    loss, lse, rows = kd.fused_kl_fwd(H, W, ids, logp, chunk, want_rows=True)
    dH, dW = kd.fused_kl_bwd(H, W, ids, logp, lse, chunk, 1.0 / T)
    torch.cuda.synchronize()
    assert abs(a["loss"] - loss.item()) <= 1e-5 * abs(loss.item())
    np.testing.assert_allclose(a["lse"], lse.cpu().numpy(), rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(a["rows"], rows.cpu().numpy(), rtol=1e-4, atol=1e-5)
    assert frob(a["dH"], dH.cpu().numpy()) <= 5e-3
    assert frob(a["dW"], dW.cpu().numpy()) <= 5e-3


@pytest.mark.parametrize("T,d,V,K,chunk", [
    (1100, 264, 1000, 7, 128),    # ragged T, d, V; three groups of four chunks, the last ragged
    (129, 72, 4099, 33, 64),
    (64, 520, 257, 5, 64),        # V = one full vocabulary tile + 1
    (77, 8, 31, 3, 16),           # tiny d and V
    (600, 128, 3000, 16, 2048),   # one group shorter than the chunk
    (300, 960, 1000, 7, 128),     # d a multiple of 480, not of 512: dW in 480-wide tiles
])
def test_ragged_shapes_match_oracle(cuda_dev, T, d, V, K, chunk):
    H, W = synth.student(T, d, V, seed=T * 7 + d)
    ids, logp = synth.synthetic_cache(T, V, K, seed=V)
    # ids on vocabulary-tile edges and at both ends of the vocabulary
    for t in range(0, T, 3):
        row = ids[t].tolist()
        for e in [0, V - 1, 255 % V, 256 % V, 511 % V]:
            if e not in row:
                row[np.random.default_rng(t + e).integers(K)] = e
        ids[t] = torch.tensor(row, dtype=torch.int32)
    H, W, ids, logp = H.to(cuda_dev), W.to(cuda_dev), ids.to(cuda_dev), logp.to(cuda_dev)
    compare(one_call(H, W, ids, logp, chunk), oracle_run(H, W, ids, logp))


def test_K_equals_V_and_duplicates(cuda_dev):
    c = synth.CONFIGS["tiny"]
    T, d, V = 128, c["d"], c["V"]
    H, W = synth.student(T, d, V, c["seed"])
    tl = synth.teacher_logits(H, W, c["seed"])
    ids, logp = O.topk_cache(tl.numpy(), V)
    H, W = H.to(cuda_dev), W.to(cuda_dev)
    ids, logp = torch.from_numpy(ids).to(cuda_dev), torch.from_numpy(logp).to(cuda_dev)
    compare(one_call(H, W, ids, logp, 64), oracle_run(H, W, ids, logp))
    T, d, V, K = 96, 128, 700, 6
    H, W = synth.student(T, d, V, seed=11)
    ids, logp = synth.synthetic_cache(T, V, K, seed=12)
    ids[:, 1] = ids[:, 0]
    H, W, ids, logp = H.to(cuda_dev), W.to(cuda_dev), ids.to(cuda_dev), logp.to(cuda_dev)
    compare(one_call(H, W, ids, logp, 64), oracle_run(H, W, ids, logp))


def test_grad_scale_and_accumulate(cuda_dev):
    H, W, ids, logp, chunk = tiny_inputs(cuda_dev)
    T = H.shape[0]
    a = one_call(H, W, ids, logp, chunk)
    two = torch.tensor(2.0, device=cuda_dev)
    b = one_call(H, W, ids, logp, chunk, grad_scale_dev=two)
    assert frob(b["dH"], 2 * a["dH"]) <= 1e-2 and frob(b["dW"], 2 * a["dW"]) <= 1e-2
    dW = torch.from_numpy(a["dW"]).to(cuda_dev)
    kd.fused_kl_fwdbwd(H, W, ids, logp, chunk, 1.0 / T, dW=dW, accumulate_dW=True)
    torch.cuda.synchronize()
    assert frob(dW.cpu().numpy(), 2 * a["dW"]) <= 1e-5


@pytest.mark.parametrize("name", ["llama3b", "gptoss20b"])
def test_full_width_truncated_run(cuda_dev, gemm_tiles, name):
    """Full d, V and chunk of the workloads, T = one full group of chunks
    plus a ragged second group of 37 positions (G = clamp(4096 / chunk, 1, 4)
    as include/kd.h states): every element of dW and dH against the
    oracle."""
    if gemm_tiles != ("1", None):
        pytest.skip("full-width check runs in the default tile configuration")
    c = synth.CONFIGS[name]
    chunk = c["chunk"]
    G = min(4, max(1, 4096 // chunk))
    Tp = G * chunk + 37
    H, W = synth.student(Tp, c["d"], c["V"], c["seed"], device=cuda_dev)
    ids, logp = synth.synthetic_cache(Tp, c["V"], c["K"], c["seed"])
    ids, logp = ids.to(cuda_dev), logp.to(cuda_dev)
    g = one_call(H, W, ids, logp, chunk)
    H64 = H.float().cpu().numpy().astype(np.float64)
    W64 = W.float().cpu().numpy().astype(np.float64)
    idn, lpn = ids.cpu().numpy(), logp.cpu().numpy()
    dW_o = np.zeros_like(W64)
    dH_o = np.empty_like(H64)
    L_o = np.empty(Tp)
    for t0 in range(0, Tp, 256):
        t1 = min(Tp, t0 + 256)
        z = O.student_logits(H64[t0:t1], W64)
        L_o[t0:t1] = O.kl_rows_from_logits(z, idn[t0:t1], lpn[t0:t1])[0]
        gz = O.dlogits(z, idn[t0:t1], lpn[t0:t1], 1.0 / Tp)
        dW_o += gz.T @ H64[t0:t1]
        dH_o[t0:t1] = gz @ W64
    assert abs(g["loss"] - L_o.mean()) <= LOSS_RTOL * abs(L_o.mean())
    np.testing.assert_allclose(g["rows"], L_o, rtol=LOSS_RTOL, atol=1e-4)
    assert frob(g["dW"], dW_o) <= GRAD_RTOL
    assert frob(g["dW"], dW_o) <= GRAD_ACHIEVED
    assert frob(g["dH"], dH_o) <= GRAD_RTOL
    assert frob(g["dH"], dH_o) <= GRAD_ACHIEVED
