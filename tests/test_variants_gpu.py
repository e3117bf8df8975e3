"""The loss variants of kd_kl_options (temperature, position mask, mean over
the included positions, bf16 dH) through the forward, backward, single-call
and autograd paths, against the fp64 oracle's tempered and masked
definitions on the same seeded inputs. Tolerances as for the plain loss:
loss relative 1e-3, dH and dW relative Frobenius 1e-2."""

import numpy as np
import pytest
import torch

import top_kl_loss_tcgen05_b300 as kd
from oracle import kd_oracle as O
from top_kl_loss_tcgen05_b300 import _native, synth

pytestmark = pytest.mark.gpu

LOSS_RTOL = 1e-3
GRAD_RTOL = 1e-2


def frob(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def inputs(dev, T=256, d=256, V=4096, K=16, seed=1000):
    H, W = synth.student(T, d, V, seed)
    tl = synth.teacher_logits(H, W, seed)
    ids, logp = O.topk_cache(tl.numpy(), K)
    return H.to(dev), W.to(dev), torch.from_numpy(ids).to(dev), torch.from_numpy(logp).to(dev)


def oracle(H, W, ids, logp, tau=1.0, mask=None, over=False):
    Hn, Wn = H.float().cpu().numpy(), W.float().cpu().numpy()
    i, lp = ids.cpu().numpy(), logp.cpu().numpy()
    m = None if mask is None else mask.cpu().numpy()
    loss, lse, L = O.fused_kl_forward(Hn, Wn, i, lp, temperature=tau, mask=m, mean_over_mask=over)
    T = Hn.shape[0]
    n = T if (m is None or not over) else int((m != 0).sum())
    dH, dW = O.fused_kl_backward(Hn, Wn, i, lp, (1.0 / n) if n else 0.0, temperature=tau, mask=m)
    return loss, lse, L, dH, dW


def make_mask(T, dev, seed=3, frac=0.7):
    g = torch.Generator().manual_seed(seed)
    m = (torch.rand(T, generator=g) < frac).to(torch.uint8)
    m[0], m[T - 1] = 1, 0
    return m.to(dev)


def check(loss, lse, rows, dH, dW, ref):
    lo, lse_o, L_o, dH_o, dW_o = ref
    assert abs(loss - lo) <= LOSS_RTOL * abs(lo), (loss, lo)
    np.testing.assert_allclose(lse, lse_o, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(rows, L_o, rtol=1e-3, atol=2e-4)
    assert frob(dH, dH_o) <= GRAD_RTOL
    assert frob(dW, dW_o) <= GRAD_RTOL


@pytest.mark.parametrize("tau", [0.5, 2.0])
def test_temperature_fwd_bwd_and_single_call(cuda_dev, tau):
    H, W, ids, logp = inputs(cuda_dev)
    T = H.shape[0]
    ref = oracle(H, W, ids, logp, tau=tau)
    loss, lse, rows = kd.fused_kl_fwd(H, W, ids, logp, 64, want_rows=True, temperature=tau)
    dH, dW = kd.fused_kl_bwd(H, W, ids, logp, lse, 64, 1.0 / T, temperature=tau)
    torch.cuda.synchronize()
    check(loss.item(), lse.cpu().numpy(), rows.cpu().numpy(), dH.cpu().numpy(), dW.cpu().numpy(), ref)
    l2, lse2, r2, dH2, dW2 = kd.fused_kl_fwdbwd(H, W, ids, logp, 64, want_rows=True, temperature=tau)
    torch.cuda.synchronize()
    check(l2.item(), lse2.cpu().numpy(), r2.cpu().numpy(), dH2.cpu().numpy(), dW2.cpu().numpy(), ref)


@pytest.mark.parametrize("over", [False, True])
def test_mask_fwd_bwd_and_single_call(cuda_dev, over):
    H, W, ids, logp = inputs(cuda_dev)
    T = H.shape[0]
    mask = make_mask(T, cuda_dev)
    ref = oracle(H, W, ids, logp, mask=mask, over=over)
    loss, lse, rows = kd.fused_kl_fwd(H, W, ids, logp, 64, want_rows=True, mask=mask, mean_over_mask=over)
    # grad_scale: 1/T carries the mean over T; over the mask the library applies 1/N
    dH, dW = kd.fused_kl_bwd(H, W, ids, logp, lse, 64, 1.0 if over else 1.0 / T, mask=mask, mean_over_mask=over)
    torch.cuda.synchronize()
    dHn = dH.cpu().numpy()
    excluded = mask.cpu().numpy() == 0
    assert np.all(dHn[excluded] == 0.0) and np.all(rows.cpu().numpy()[excluded] == 0.0)
    check(loss.item(), lse.cpu().numpy(), rows.cpu().numpy(), dHn, dW.cpu().numpy(), ref)
    l2, lse2, r2, dH2, dW2 = kd.fused_kl_fwdbwd(H, W, ids, logp, 64, want_rows=True, mask=mask, mean_over_mask=over)
    torch.cuda.synchronize()
    check(l2.item(), lse2.cpu().numpy(), r2.cpu().numpy(), dH2.cpu().numpy(), dW2.cpu().numpy(), ref)


def test_temperature_and_mask_on_ragged_shapes(cuda_dev):
    T, d, V, K, chunk, tau = 300, 264, 1000, 7, 128, 1.7
    H, W = synth.student(T, d, V, seed=77)
    ids, logp = synth.synthetic_cache(T, V, K, seed=78)
    H, W, ids, logp = H.to(cuda_dev), W.to(cuda_dev), ids.to(cuda_dev), logp.to(cuda_dev)
    mask = make_mask(T, cuda_dev, seed=9)
    ref = oracle(H, W, ids, logp, tau=tau, mask=mask, over=True)
    l, lse, r, dH, dW = kd.fused_kl_fwdbwd(H, W, ids, logp, chunk, want_rows=True, temperature=tau, mask=mask,
                                           mean_over_mask=True)
    torch.cuda.synchronize()
    check(l.item(), lse.cpu().numpy(), r.cpu().numpy(), dH.cpu().numpy(), dW.cpu().numpy(), ref)
    loss, lse, rows = kd.fused_kl_fwd(H, W, ids, logp, chunk, want_rows=True, temperature=tau, mask=mask,
                                      mean_over_mask=True)
    dH, dW = kd.fused_kl_bwd(H, W, ids, logp, lse, chunk, 1.0, temperature=tau, mask=mask, mean_over_mask=True)
    torch.cuda.synchronize()
    check(loss.item(), lse.cpu().numpy(), rows.cpu().numpy(), dH.cpu().numpy(), dW.cpu().numpy(), ref)


def test_bf16_dH(cuda_dev):
    H, W, ids, logp = inputs(cuda_dev)
    T = H.shape[0]
    ref = oracle(H, W, ids, logp)
    _, lse, _ = kd.fused_kl_fwd(H, W, ids, logp, 64)
    dH32, dW32 = kd.fused_kl_bwd(H, W, ids, logp, lse, 64, 1.0 / T)
    dHb, dWb = kd.fused_kl_bwd(H, W, ids, logp, lse, 64, 1.0 / T, dH_bf16=True)
    torch.cuda.synchronize()
    assert dHb.dtype == torch.bfloat16
    assert torch.equal(dHb, dH32.to(torch.bfloat16))  # the same fp32 accumulators, rounded once
    assert torch.equal(dWb, dW32)
    assert frob(dHb.float().cpu().numpy(), ref[3]) <= GRAD_RTOL
    _, _, _, dH1, _ = kd.fused_kl_fwdbwd(H, W, ids, logp, 64, dH_bf16=True)
    torch.cuda.synchronize()
    assert dH1.dtype == torch.bfloat16 and frob(dH1.float().cpu().numpy(), ref[3]) <= GRAD_RTOL


def test_all_positions_masked(cuda_dev):
    H, W, ids, logp = inputs(cuda_dev, T=128)
    mask = torch.zeros(128, dtype=torch.uint8, device=cuda_dev)
    l, _, r, dH, dW = kd.fused_kl_fwdbwd(H, W, ids, logp, 64, want_rows=True, mask=mask, mean_over_mask=True)
    torch.cuda.synchronize()
    assert l.item() == 0.0 and torch.all(r == 0) and torch.all(dH == 0) and torch.all(dW == 0)


def test_autograd_with_temperature_and_mask(cuda_dev):
    H, W, ids, logp = inputs(cuda_dev)
    mask = make_mask(H.shape[0], cuda_dev, seed=4).bool()
    ref = oracle(H, W, ids, logp, tau=2.0, mask=mask.to(torch.uint8), over=True)
    Hg = H.clone().requires_grad_(True)
    Wg = W.clone().requires_grad_(True)
    loss = kd.FusedKL.apply(Hg, Wg, ids, logp, 64, 2.0, mask, True)
    (3.0 * loss).backward()
    assert abs(loss.item() - ref[0]) <= LOSS_RTOL * abs(ref[0])
    assert Hg.grad.dtype == torch.bfloat16
    assert frob(Hg.grad.float().cpu().numpy(), 3.0 * ref[3]) <= GRAD_RTOL
    assert frob(Wg.grad.float().cpu().numpy(), 3.0 * ref[4]) <= GRAD_RTOL


@pytest.mark.parametrize("tau,over,bf", [(0.0, 0, 0), (-1.0, 0, 0), (float("inf"), 0, 0), (1.0, 2, 0), (1.0, 0, 3)])
def test_invalid_options_are_rejected_before_launch(cuda_dev, tau, over, bf):
    H, W, ids, logp = inputs(cuda_dev, T=64)
    ws = kd.fused_kl_workspace(256, 4096, 16, 64, cuda_dev)
    o = _native.KLOptions(tau, None, over, bf)
    out = torch.empty(64, device=cuda_dev)
    import ctypes
    rc = _native.lib().kd_fused_kl_fwd_ex(H.data_ptr(), W.data_ptr(), ids.data_ptr(), logp.data_ptr(), 64, 256, 4096,
                                          16, 64, out.data_ptr(), out.data_ptr(), None, ctypes.byref(o),
                                          ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert rc == 1
