"""Position-sharded data parallelism with libkd's kernels on one GPU.

Each shard runs the real loss path with the 1 / T_global gradient scale.
Without collectives (one process, one GPU), the shards' results are summed
here as the all-reduce would sum them, and must match the full-batch call and
the oracle. A one-rank NCCL group then runs the helper and the autograd
Function with their collectives on the device."""

import os
import socket

import numpy as np
import pytest
import torch

import top_kl_loss_tcgen05_b300 as kd
from oracle import kd_oracle as O
from top_kl_loss_tcgen05_b300 import dp, synth

pytestmark = pytest.mark.gpu


def frob(a, b):
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(np.asarray(a, np.float64) - b) / np.linalg.norm(b))


def _inputs(dev, T=301, d=128, V=3000, K=12, seed=41):
    H, W = synth.student(T, d, V, seed)
    ids, logp = synth.synthetic_cache(T, V, K, seed + 1)
    return H.to(dev), W.to(dev), ids.to(dev), logp.to(dev)


def test_shards_summed_match_the_full_batch_and_the_oracle(cuda_dev):
    H, W, ids, logp = _inputs(cuda_dev)
    T = H.shape[0]
    chunk = 64
    parts = []
    for r in range(3):
        t0, t1 = dp.shard_range(T, 3, r)
        parts.append(dp.dp_fused_kl_step(H[t0:t1], W, ids[t0:t1], logp[t0:t1], chunk, T))
    loss = sum(float(p[0]) for p in parts)
    dW = sum(p[2] for p in parts)
    dH = torch.cat([p[1] for p in parts])
    l_full, _, _, dH_full, dW_full = kd.fused_kl_fwdbwd(H, W, ids, logp, chunk)
    torch.cuda.synchronize()
    assert abs(loss - l_full.item()) <= 1e-5 * abs(l_full.item())
    assert torch.equal(dH, dH_full)  # per-position: independent of the sharding
    assert frob(dW.cpu().numpy(), dW_full.cpu().numpy()) <= 1e-5
    Hn, Wn = H.float().cpu().numpy(), W.float().cpu().numpy()
    lo, _, _ = O.fused_kl_forward(Hn, Wn, ids.cpu().numpy(), logp.cpu().numpy())
    dH_o, dW_o = O.fused_kl_backward(Hn, Wn, ids.cpu().numpy(), logp.cpu().numpy(), 1.0 / T)
    assert abs(loss - lo) <= 1e-3 * abs(lo)
    assert frob(dH.cpu().numpy(), dH_o) <= 1e-2
    assert frob(dW.cpu().numpy(), dW_o) <= 1e-2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_one_rank_nccl_group_runs_the_collectives_on_the_device(cuda_dev):
    import torch.distributed as dist

    if dist.is_initialized():
        pytest.skip("a process group is already initialised")
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=cuda_dev)
    try:
        pg = dist.new_group([0])
        H, W, ids, logp = _inputs(cuda_dev, T=200)
        T = H.shape[0]
        loss, dH, dW = dp.dp_fused_kl_step(H, W, ids, logp, 64, T, process_group=pg)
        l_full, _, _, dH_full, dW_full = kd.fused_kl_fwdbwd(H, W, ids, logp, 64)
        torch.cuda.synchronize()
        assert abs(loss.item() - l_full.item()) <= 1e-6 * abs(l_full.item())
        assert torch.equal(dH, dH_full) and torch.equal(dW, dW_full)
        # autograd: the recompute backward with the upstream gradient on the device
        Hg = H.clone().requires_grad_(True)
        Wg = W.clone().requires_grad_(True)
        lg = dp.DPFusedKL.apply(Hg, Wg, ids, logp, 64, T, pg)
        (2.0 * lg).backward()
        torch.cuda.synchronize()
        assert abs(lg.item() - l_full.item()) <= 1e-5 * abs(l_full.item())
        assert frob(Hg.grad.float().cpu().numpy(), 2.0 * dH_full.cpu().numpy()) <= 1e-2
        assert frob(Wg.grad.float().cpu().numpy(), 2.0 * dW_full.cpu().numpy()) <= 1e-2
        # a rank without positions (more ranks than positions): zeros, no libkd
        # call (libkd refuses T = 0), and both all-reduces still run
        He, ide, lpe = H[:0], ids[:0], logp[:0]
        loss_e, dH_e, dW_e = dp.dp_fused_kl_step(He, W, ide, lpe, 64, T, process_group=pg)
        torch.cuda.synchronize()
        assert loss_e.item() == 0.0 and dH_e.shape == (0, H.shape[1]) and dW_e.dtype == torch.float32
        assert dW_e.device == W.device and not dW_e.any()
        He_g = He.clone().requires_grad_(True)
        We_g = W.clone().requires_grad_(True)
        le = dp.DPFusedKL.apply(He_g, We_g, ide, lpe, 64, T, pg)
        le.backward()
        torch.cuda.synchronize()
        assert le.item() == 0.0 and He_g.grad.shape == He.shape and not We_g.grad.any()
    finally:
        dist.destroy_process_group()
