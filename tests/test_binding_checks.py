"""The Python binding refuses tensors it cannot pass to the CUDA library
(CPU): wrong dtype, not on a CUDA device, wrong shape. There is no CPU
fallback, so a CPU tensor is an error, never a slow path."""

import pytest
import torch

import top_kl_loss_tcgen05_b300 as kd


def _cpu_inputs(T=8, d=16, V=32, K=4):
    H = torch.zeros(T, d, dtype=torch.bfloat16)
    W = torch.zeros(V, d, dtype=torch.bfloat16)
    ids = torch.zeros(T, K, dtype=torch.int32)
    logp = torch.zeros(T, K, dtype=torch.float32)
    return H, W, ids, logp


def test_cpu_tensors_are_refused():
    H, W, ids, logp = _cpu_inputs()
    with pytest.raises(ValueError, match="CUDA"):
        kd.fused_kl_fwd(H, W, ids, logp, 4)
    with pytest.raises(ValueError, match="CUDA"):
        kd.fused_kl_fwdbwd(H, W, ids, logp, 4)
    with pytest.raises(ValueError, match="CUDA"):
        kd.fused_kl_bwd(H, W, ids, logp, torch.zeros(8), 4, 0.125)
    with pytest.raises(ValueError, match="CUDA"):
        kd.topk_cache(torch.zeros(4, 32), 4)
    with pytest.raises(ValueError, match="CUDA"):
        kd.teacher_topk_cache(H, W, 4)
    with pytest.raises(ValueError, match="CUDA"):
        kd.FusedKL.apply(H, W, ids, logp, 4)


def test_wrong_dtypes_and_shapes_are_refused():
    H, W, ids, logp = _cpu_inputs()
    with pytest.raises(TypeError):
        kd.fused_kl_fwd(H.float(), W, ids, logp, 4)  # H must be bf16
    # later arguments are checked after H, whose device is wrong here: any refusal will do
    with pytest.raises((TypeError, ValueError)):
        kd.fused_kl_fwd(H, W, ids.long(), logp, 4)  # ids must be int32
    with pytest.raises((TypeError, ValueError)):
        kd.fused_kl_fwd(H, W, ids, logp.double(), 4)
    with pytest.raises(TypeError):
        kd.topk_cache(torch.zeros(4, 32, dtype=torch.float16), 4)  # bf16 or fp32 only
    with pytest.raises(ValueError):
        kd.topk_cache(torch.zeros(32), 4)  # not [T, V]
