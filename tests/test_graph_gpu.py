"""The loss calls are stream-ordered (memsets, kernel and cluster launches on
the caller's stream), so a training step can be captured once in a CUDA
graph and replayed. Replays give bitwise the eager results."""

import pytest
import torch

import top_kl_loss_tcgen05_b300 as kd
from oracle import kd_oracle as O
from top_kl_loss_tcgen05_b300 import synth

pytestmark = pytest.mark.gpu


def _inputs(dev):
    c = synth.CONFIGS["tiny"]
    H, W = synth.student(c["T"], c["d"], c["V"], c["seed"])
    tl = synth.teacher_logits(H, W, c["seed"])
    ids, logp = O.topk_cache(tl.numpy(), c["K"])
    return H.to(dev), W.to(dev), torch.from_numpy(ids).to(dev), torch.from_numpy(logp).to(dev), c["chunk"]


def test_fwd_bwd_and_single_call_replay_bitwise(cuda_dev):
    H, W, ids, logp, chunk = _inputs(cuda_dev)
    T = H.shape[0]
    ws = kd.fused_kl_workspace(H.shape[1], W.shape[0], ids.shape[1], chunk, cuda_dev)
    # eager references (also the first call on this device: attribute set-up happens here)
    loss0, lse0, _ = kd.fused_kl_fwd(H, W, ids, logp, chunk, ws=ws)
    dH0, dW0 = kd.fused_kl_bwd(H, W, ids, logp, lse0, chunk, 1.0 / T, ws=ws)
    l1, lse1, _, dH1, dW1 = kd.fused_kl_fwdbwd(H, W, ids, logp, chunk, ws=ws)
    torch.cuda.synchronize()
    ref = [t.clone() for t in (loss0, lse0, dH0, dW0, l1, lse1, dH1, dW1)]

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            loss, lse, _ = kd.fused_kl_fwd(H, W, ids, logp, chunk, ws=ws)
            dH, dW = kd.fused_kl_bwd(H, W, ids, logp, lse, chunk, 1.0 / T, ws=ws)
            la, lsea, _, dHa, dWa = kd.fused_kl_fwdbwd(H, W, ids, logp, chunk, ws=ws)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        g.replay()
        torch.cuda.synchronize()
        got = (loss, lse, dH, dW, la, lsea, dHa, dWa)
        for a, b in zip(got, ref):
            assert torch.equal(a, b)
    assert kd.read_device_status(ws) == 0
