"""Device memory of the fused loss: the library allocates nothing itself
(its only scratch is the caller's workspace, whose size does not depend on
T), and the Python calls allocate exactly their outputs. So the memory a
step needs is the inputs, the outputs and one O(chunk * V) workspace: it
grows linearly in T with the per-position bytes of H, the cache, lse and dH,
and no T x V buffer ever exists."""

import pytest
import torch

import top_kl_loss_tcgen05_b300 as kd
from top_kl_loss_tcgen05_b300 import synth

pytestmark = pytest.mark.gpu

d, V, K, chunk = 512, 32000, 32, 256


def _inputs(T, dev):
    H, W = synth.student(T, d, V, 77, device=dev)
    ids, logp = synth.synthetic_cache(T, V, K, 78)
    return H, W, ids.to(dev), logp.to(dev)


def _step(H, W, ids, logp, ws):
    T = H.shape[0]
    loss, lse, rows = kd.fused_kl_fwd(H, W, ids, logp, chunk, ws=ws, want_rows=True)
    dH, dW = kd.fused_kl_bwd(H, W, ids, logp, lse, chunk, 1.0 / T, ws=ws)
    return loss, lse, rows, dH, dW


def test_library_allocates_no_device_memory(cuda_dev):
    H, W, ids, logp = _inputs(2048, cuda_dev)
    ws = kd.fused_kl_workspace(d, V, K, chunk, cuda_dev)
    x = synth.topk_logits(512, V, 5, device=cuda_dev)
    tws = kd.workspace(256, cuda_dev)
    for _ in range(2):  # load every kernel and fill torch's cache for the outputs
        out = _step(H, W, ids, logp, ws)
        out1 = kd.fused_kl_fwdbwd(H, W, ids, logp, chunk, ws=ws)
        t = kd.topk_cache(x, K, ws=tws)
        torch.cuda.synchronize()
        del out, out1, t
    free0, _ = torch.cuda.mem_get_info(cuda_dev)
    out = _step(H, W, ids, logp, ws)
    out1 = kd.fused_kl_fwdbwd(H, W, ids, logp, chunk, ws=ws)
    t = kd.topk_cache(x, K, ws=tws)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(cuda_dev)
    assert free1 == free0
    assert kd.read_device_status(ws) == 0


def _rounded(nbytes):
    return (nbytes + 511) // 512 * 512  # torch's allocation granularity


@pytest.mark.parametrize("T", [1000, 2048, 5000])
def test_calls_allocate_exactly_their_outputs(cuda_dev, T):
    H, W, ids, logp = _inputs(T, cuda_dev)
    ws = kd.fused_kl_workspace(d, V, K, chunk, cuda_dev)
    assert ws.numel() == kd.fused_kl_workspace(d, V, K, chunk, cuda_dev).numel()  # no T in the size
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats(cuda_dev)
    before = torch.cuda.memory_allocated(cuda_dev)
    out = _step(H, W, ids, logp, ws)
    torch.cuda.synchronize()
    peak = torch.cuda.max_memory_allocated(cuda_dev) - before
    # loss (scalar), lse [T], loss_rows [T], dH [T, d] and dW [V, d], all fp32
    expect = _rounded(4) + 2 * _rounded(4 * T) + _rounded(4 * T * d) + _rounded(4 * V * d)
    assert peak == expect, (peak, expect)
    assert sum(_rounded(o.numel() * o.element_size()) for o in out) == expect
