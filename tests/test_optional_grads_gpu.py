"""Skipping a gradient: dH = NULL or dW = NULL in kd_fused_kl_bwd(_ex) and
kd_fused_kl_fwdbwd(_ex) (want_dH / want_dW in the binding; autograd's
needs_input_grad in FusedKL). The skipped gradient's GEMM tiles are not
launched, and the other gradient must be bitwise the one the full call
computes: its tiles, their operands and their order do not change."""

import pytest
import torch

import top_kl_loss_tcgen05_b300 as kd
from top_kl_loss_tcgen05_b300 import synth

pytestmark = pytest.mark.gpu


def _inputs(dev, T, d, V, K, seed):
    H, W = synth.student(T, d, V, seed)
    ids, logp = synth.synthetic_cache(T, V, K, seed + 1)
    return H.to(dev), W.to(dev), ids.to(dev), logp.to(dev)


# d = 960: the 480-wide dW tiles; T = 300 with chunk 64: five groups, a ragged last one
SHAPES = [(300, 256, 4096, 16, 64), (300, 960, 3000, 8, 64)]


@pytest.mark.parametrize("T,d,V,K,chunk", SHAPES)
@pytest.mark.parametrize("dH_bf16", [False, True])
def test_backward_computes_only_what_is_asked(cuda_dev, T, d, V, K, chunk, dH_bf16):
    H, W, ids, logp = _inputs(cuda_dev, T, d, V, K, 11)
    _, lse, _ = kd.fused_kl_fwd(H, W, ids, logp, chunk)
    dH, dW = kd.fused_kl_bwd(H, W, ids, logp, lse, chunk, 1.0 / T, dH_bf16=dH_bf16)
    dH_only, none_w = kd.fused_kl_bwd(H, W, ids, logp, lse, chunk, 1.0 / T, dH_bf16=dH_bf16, want_dW=False)
    none_h, dW_only = kd.fused_kl_bwd(H, W, ids, logp, lse, chunk, 1.0 / T, dH_bf16=dH_bf16, want_dH=False)
    torch.cuda.synchronize()
    assert none_w is None and none_h is None
    assert torch.equal(dH_only, dH)
    assert torch.equal(dW_only, dW)
    # accumulation into an existing dW, without dH. The group partials are
    # reduce-added onto dW one group at a time, which rounds differently from
    # doubling the finished sum: a few fp32 ulps of the partial sums, which
    # can exceed the final value where the groups' contributions cancel, so
    # the absolute bound scales with dW's magnitude.
    acc = dW.clone()
    _, acc = kd.fused_kl_bwd(H, W, ids, logp, lse, chunk, 1.0 / T, dW=acc, accumulate_dW=True, want_dH=False)
    torch.cuda.synchronize()
    assert torch.allclose(acc, 2 * dW, rtol=1e-5, atol=1e-6 * dW.abs().max().item())
    with pytest.raises(ValueError):
        kd.fused_kl_bwd(H, W, ids, logp, lse, chunk, 1.0 / T, want_dH=False, want_dW=False)


@pytest.mark.parametrize("T,d,V,K,chunk", SHAPES)
def test_single_call_computes_only_what_is_asked(cuda_dev, T, d, V, K, chunk):
    H, W, ids, logp = _inputs(cuda_dev, T, d, V, K, 12)
    loss, lse, _, dH, dW = kd.fused_kl_fwdbwd(H, W, ids, logp, chunk)
    l1, lse1, _, dH1, w1 = kd.fused_kl_fwdbwd(H, W, ids, logp, chunk, want_dW=False)
    l2, lse2, _, h2, dW2 = kd.fused_kl_fwdbwd(H, W, ids, logp, chunk, want_dH=False)
    torch.cuda.synchronize()
    assert w1 is None and h2 is None
    assert torch.equal(l1, loss) and torch.equal(l2, loss) and torch.equal(lse1, lse) and torch.equal(lse2, lse)
    assert torch.equal(dH1, dH)
    assert torch.equal(dW2, dW)


def test_autograd_skips_the_frozen_side(cuda_dev):
    T, d, V, K, chunk = 300, 256, 4096, 16, 64
    H, W, ids, logp = _inputs(cuda_dev, T, d, V, K, 13)
    Hf, Wf = H.clone().requires_grad_(True), W.clone().requires_grad_(True)
    kd.FusedKL.apply(Hf, Wf, ids, logp, chunk).backward()
    # frozen LM head: only H gets a gradient, and it is the full run's
    Hh, Wh = H.clone().requires_grad_(True), W.clone()
    kd.FusedKL.apply(Hh, Wh, ids, logp, chunk).backward()
    # frozen body: only W
    Hw, Ww = H.clone(), W.clone().requires_grad_(True)
    kd.FusedKL.apply(Hw, Ww, ids, logp, chunk).backward()
    torch.cuda.synchronize()
    assert Wh.grad is None and Hw.grad is None
    assert torch.equal(Hh.grad, Hf.grad)
    assert torch.equal(Ww.grad, Wf.grad)
